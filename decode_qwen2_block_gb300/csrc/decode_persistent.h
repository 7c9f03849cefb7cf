// Persistent decode kernel: one launch runs one decode token through a stack
// of blocks (see decode_persistent.cu).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace blk {

constexpr int kDecMaxLayers = 32;  // layers per launch (the host loops beyond)
constexpr int kDecMaxVec = 12288;  // longest input vector a phase stages (elements)

struct DecLayer {
  const __half *wq, *wk, *wv, *bq, *bk, *bv, *wo, *ln1, *ln2, *wg, *wu, *wd;
  __half* kc;      // [Hkv, max_ctx, D]
  __half* vc;
  __half* k_new;   // [Hkv, D] or null
  __half* v_new;
};

struct DecodeParams {
  CUtensorMap tm_k[kDecMaxLayers];  // cache viewed as [Hkv * max_ctx, D], box 64 x 64, SW128
  CUtensorMap tm_v[kDecMaxLayers];
  DecLayer layer[kDecMaxLayers];
  int n_layers;
  int H, Hq, Hkv, D, I;
  float eps;
  float scale_log2;     // log2(e) / sqrt(D)
  int64_t max_ctx;
  int64_t cache_len;    // slot of the new token
  const int64_t* pos;   // [1]
  const float2* rope;
  int64_t rope_len;
  const __half* x_in;   // [H]
  __half* out;          // [H]
  // workspace
  __half* xbuf0;        // [H] ping-pong layer outputs
  __half* xbuf1;
  float* q32;           // [Hq * D]
  float* part;          // [Hq][S][D + 4]  (acc[D], m, l, pad): rows 16-byte aligned
  __half* attn16;       // [Hq * D]
  float* h32;           // [H]
  __half* act16;        // [I]
  unsigned* barrier;    // grid-barrier counter, zeroed before the launch
  int* err;
  int S;                // attention splits per kv head used by this launch
  int fold;             // S <= 32: splits merged in the o_proj staging
  uint64_t* trace;      // optional per-CTA phase timeline (nullptr = off)
  size_t trace_len;     // entries of trace
};

// Workspace bytes for the decode path (grid = num_sms CTAs).
size_t decode_ws_bytes(int H, int Hq, int Hkv, int D, int I, int num_sms);
// Carves the workspace and fills the workspace pointers of `p`.
void decode_ws_carve(DecodeParams& p, void* ws, int num_sms);

cudaError_t launch_decode_persistent(DecodeParams& p, int num_sms, cudaStream_t s);
cudaError_t configure_decode_persistent();

}  // namespace blk
