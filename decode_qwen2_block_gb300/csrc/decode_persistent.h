// Persistent decode kernel: one launch runs one decode token through a stack
// of blocks (see decode_persistent.cu).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace blk {

constexpr int kDecMaxLayers = 16;  // layers per launch (the host loops beyond)
constexpr int kDecMaxVec = 12288;  // longest input vector a phase stages (elements)

struct DecLayer {
  const __half *wq, *wk, *wv, *bq, *bk, *bv, *wo, *ln1, *ln2, *wg, *wu, *wd;
  __half* kc;      // [Hkv, max_ctx, D]
  __half* vc;
  __half* k_new;   // [Hkv, D] or null
  __half* v_new;
};

constexpr int kDecRoles = 7;       // wq wk wv wo w_gate w_up w_down

struct DecodeParams {
  CUtensorMap tm_k[kDecMaxLayers];  // cache viewed as [Hkv * max_ctx, D], box 64 x 64, SW128
  CUtensorMap tm_v[kDecMaxLayers];
  // weights [rows, K]: 3-D view (64, rows, K / 64) with box (64, 8, min(24, K / 64)) when
  // K % 64 == 0, else 2-D (K, rows) with box (64, 8); 128-byte swizzle either way
  CUtensorMap tm_w[kDecMaxLayers][kDecRoles];
  int w3d[kDecRoles];     // 1: tm_w of this role is the 3-D view
  int wbox_z[kDecRoles];  // 3-D box depth (column blocks)
  int wnz[kDecRoles];     // column blocks of 64 in K, rounded up
  DecLayer layer[kDecMaxLayers];
  int n_layers;
  int H, Hq, Hkv, D, I;
  float eps;
  float scale_log2;     // log2(e) / sqrt(D)
  int64_t max_ctx;
  int64_t cache_len;    // slot of the new token
  int64_t window;       // sliding window in slots (0 = attend [0, cache_len])
  const int64_t* pos;   // [1]
  const float2* rope;
  int64_t rope_len;
  const __half* x_in;   // [H]
  __half* out;          // [H]
  // workspace
  float* pdown;         // [nc_down][H] DOWN partials per 1536-column chunk
  int nc_down;
  float* q32;           // [Hq * D]
  uint8_t* part;        // [Hq][S] rows of 2D + 16 bytes: acc / sum (D fp16), (max, sum) float2
  __half* attn16;       // [Hq * D]
  float* h32;           // [H]
  __half* act16;        // [I]
  unsigned* barrier;    // grid-barrier counter, zeroed before the launch
  int* err;
  int S;                // attention splits per kv head used by this launch
  int fold;             // S <= 32: splits merged in the o_proj staging
  uint64_t* trace;      // optional per-CTA phase timeline (nullptr = off)
  size_t trace_len;     // entries of trace
  // weight format: 0 fp16 (tm_w views the fp16 matrices), 1 INT8 codes with
  // one fp16 scale per row, 2 packed int4 codes with an fp16 scale and a
  // uint8 zero point per qgroup columns of a row (tm_w views the codes)
  int fmt;
  int qgroup;
  int qgroup_lg;        // log2(qgroup): int4 groups are powers of two
  const uint16_t* qscale[kDecMaxLayers][kDecRoles];  // fp16 bits
  const uint8_t* qzero[kDecMaxLayers][kDecRoles];
};

// Workspace bytes for the decode path (grid = num_sms CTAs).
size_t decode_ws_bytes(int H, int Hq, int Hkv, int D, int I, int num_sms);
// Carves the workspace and fills the workspace pointers of `p`.
void decode_ws_carve(DecodeParams& p, void* ws, int num_sms);

static_assert(sizeof(DecodeParams) <= 32764, "kernel parameter space");

cudaError_t launch_decode_persistent(DecodeParams& p, int num_sms, cudaStream_t s);
cudaError_t configure_decode_persistent();
// Quantized formats stage a phase's scales in shared memory: the largest
// number of entries any phase needs (0 for fp16), and the limit.
int decode_q_max_entries(int H, int Hq, int Hkv, int D, int I, int fmt, int group, int num_sms);
int decode_q_entry_limit();

}  // namespace blk
