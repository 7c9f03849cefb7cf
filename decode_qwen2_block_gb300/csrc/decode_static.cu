// blk_decode_static: the decode step for callers that cannot allocate device
// memory.  Its scratch (the decode intermediates and the split-K attention
// partials and counters) lives in one file-scope __device__ array instead of
// a caller-provided workspace.
//
// Who needs this: code that runs where it may not call cudaMalloc or any
// allocating routine — e.g. a plugin inside a host framework whose memory
// manager owns every device byte and rejects outside allocations, or a
// latency-critical serving loop that must not allocate because cudaMalloc and
// cudaFree can synchronize the whole device and stall other streams.
#include <mutex>

#include "../../include/blk.h"
#include "blk_internal.h"

namespace {

// Holds the workspace of one decode call; every GPU that loads the library
// keeps this array until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[BLK_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device

// Host code cannot use g_decode_scratch as a pointer (on the host the name is
// only a stand-in for the device symbol), so look up its device address once
// per device, with that device current.
int scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return BLK_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[device]) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return BLK_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return BLK_ERR_CUDA;
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess || p == nullptr) return BLK_ERR_CUDA;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return BLK_OK;
}

}  // namespace

extern "C" int blk_decode_static(blk_handle h, const blk_weights* w, const void* x,
                                 const int64_t* pos, int64_t cache_len, void* k_cache,
                                 void* v_cache, void* out, void* k_new, void* v_new,
                                 void* stream) {
  // A missing pointer is reported before the size limit, the size limit
  // before blk_decode's own checks (shape, alignment, cache bounds).
  if (!h || !w || !x || !pos || !k_cache || !v_cache || !out) return BLK_ERR_NULL;
  if (blk_internal_decode_ws_bytes(h) > BLK_STATIC_SCRATCH_BYTES)
    return BLK_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int rc = scratch_address(blk_internal_device(h), &scratch);
  if (rc != BLK_OK) return rc;
  // Leftovers of an earlier call in the array do not matter: the only words
  // that must start at zero (the decode kernel's synchronisation counters)
  // are zeroed by a cudaMemsetAsync on the call's stream before each launch,
  // and every other region is written in full before it is read.
  return blk_decode(h, w, x, pos, cache_len, k_cache, v_cache, out, k_new, v_new, scratch,
                    BLK_STATIC_SCRATCH_BYTES, stream);
}
