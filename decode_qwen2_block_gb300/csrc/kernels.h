// Host-visible kernel parameter blocks and launchers.  The C ABI in
// blk_api.cu validates arguments, carves the workspace and calls these.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace blk {

// ---------------------------------------------------------------- decode
// Weight-streaming matrix-vector product for one token.  Modes:
//   QKV    : x16 = block input; RMSNorm(ln1) prologue; rows of wq|wk|wv in
//            RoPE pairs (i, i + D/2); epilogue adds bias, rotates q and k,
//            writes q (fp32), K/V to cache slot `slot` and k_new/v_new.
//   O      : x16 = attention output; epilogue h32 = acc + res16 (block input).
//   GATEUP : x32 = h; RMSNorm(ln2) prologue; rows j of w_gate and w_up;
//            epilogue out16 = silu(gate) * up.
//   DOWN   : x16 = SwiGLU activation; epilogue out16 = acc + res32 (h).
enum GemvMode { kGemvQKV = 0, kGemvO = 1, kGemvGateUp = 2, kGemvDown = 3 };

struct GemvParams {
  const __half* W[3];
  const __half* bias[3];
  int K;        // input length
  int N;        // QKV: unused; GATEUP: intermediate; O/DOWN: hidden
  const __half* x16;
  const float* x32;
  const __half* gain;
  float eps;
  // QKV
  int Hq, Hkv, D, parts;
  const int64_t* pos;
  const float2* rope;
  int64_t rope_len;
  __half* kc;
  __half* vc;
  int64_t max_ctx;
  int64_t slot;
  __half* k_new;
  __half* v_new;
  float* q32;
  unsigned* counters;  // zeroed by the QKV kernel for the attention combine
  int n_counters;
  // residuals / outputs
  const __half* res16;
  const float* res32;
  float* out32;
  __half* out16;
  int* err;
  // streaming geometry (set by the launcher)
  int rows_per_chunk, warps_per_row, stage_bytes, n_stages, max_rows;
};

cudaError_t launch_gemv(GemvParams p, int mode, int grid, cudaStream_t s,
                        bool pdl);
// Grid size and dynamic shared memory for a mode (used for the launch and for
// workspace sizing).
int gemv_grid(const GemvParams& p, int mode, int num_sms);

struct DecodeAttnParams {
  const float* q32;   // [Hq * D]
  const __half* kc;   // [Hkv, max_ctx, D]
  const __half* vc;
  int64_t max_ctx;
  int64_t n_keys;     // cache_len + 1
  int Hq, Hkv, D;
  int splits, slots_per_split;
  float2* part_ml;    // [Hq, splits] (max in log2 units, sum)
  float* part_acc;    // [Hq, splits, D]
  unsigned* counters; // [Hkv], zero on entry
  __half* attn16;     // [Hq * D]
  float scale_log2;   // log2(e) / sqrt(D)
  int* err;
};

cudaError_t launch_decode_attn(const DecodeAttnParams& p, cudaStream_t s,
                               bool pdl);
void decode_attn_splits(int64_t n_keys, int Hkv, int num_sms, int* splits,
                        int* slots_per_split);
int decode_attn_max_splits(int64_t max_ctx, int Hkv, int num_sms);

// --------------------------------------------------------------- prefill
cudaError_t launch_rmsnorm_rows(const void* x, bool x_is_f32, const __half* g,
                                int rows, int H, float eps, __half* y,
                                cudaStream_t s, bool pdl);

struct PrefillAttnParams {
  const __half* q16;  // [T, Hq, D]
  const __half* kc;
  const __half* vc;
  int64_t max_ctx, cache_len;
  int T, Hq, Hkv, D;
  float scale_log2;
  __half* attn16;  // [T, Hq * D]
};
cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t s,
                                bool pdl);

// Sets the per-kernel shared-memory limits (called once per device).
cudaError_t configure_kernels();

}  // namespace blk
