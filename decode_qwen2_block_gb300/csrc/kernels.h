// Host-visible kernel parameter blocks and launchers.  The C ABI in
// blk_api.cu validates arguments, carves the workspace and calls these.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace blk {

// --------------------------------------------------------------- prefill
cudaError_t launch_rmsnorm_rows(const void* x, bool x_is_f32, const __half* g,
                                int rows, int H, float eps, __half* y,
                                cudaStream_t s, bool pdl);
// h32 = sum_s part[s] (s ascending) + res16, y = RMSNorm(h32) * g (rows of
// width H, part = S <= 8 partials [rows][H] fp32).
// Down split-K reduction fused with the next layer's RMSNorm (layer stacks):
// out16 = fp16(sum of S partials [S][rows][H] + res32) and y = RMSNorm(out16)
// * g, bit-identical to launch_splitk_reduce followed by launch_rmsnorm_rows
// on out16.  S <= 16, H a multiple of 8.
cudaError_t launch_splitk_reduce_norm(const float* part, int S, const float* res32,
                                      __half* out16, const __half* g, int rows, int H, float eps,
                                      __half* y, cudaStream_t s);
cudaError_t launch_rmsnorm_splitk(const float* part, int S, const __half* res16, float* h32,
                                  const __half* g, int rows, int H, float eps, __half* y,
                                  cudaStream_t s, bool pdl);

struct PrefillAttnParams {
  CUtensorMap tm_q;   // q [T, Hq, D] viewed as (D, Hq, T), box 64 x 1 x 128, SW128
  CUtensorMap tm_k;   // K cache viewed as (D, L + T, Hkv), box 64 x 128 x 1, SW128:
  CUtensorMap tm_v;   //   slots past L + T read as zeros
  const __half* q16;  // [T, Hq, D]
  int64_t max_ctx, cache_len;
  int T, Hq, Hkv, D;
  float scale_log2;   // log2(e) / sqrt(D)
  int64_t window;     // sliding window in slots (0 = full causal attention)
  __half* attn16;  // [T, Hq * D]
  // Split of each 128-row block's tiles into chunks of chunk_tiles (one CTA
  // each; grid (Hq, nqb, grid_chunks)), set by plan_prefill_attn.  Blocks with
  // more than one chunk leave partials in `part` ([Hq][nqb][max_chunks] slots,
  // prefill_attn_part_bytes) for launch_attn_merge.
  int nqb, chunk_tiles, grid_chunks, max_chunks;
  float* part;
  int* err;
};
int prefill_attn_max_chunks(int64_t T, int Hq, int num_sms);
size_t prefill_attn_part_bytes(int64_t T, int Hq, int D, int num_sms);
void plan_prefill_attn(PrefillAttnParams& p, int num_sms);
cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t s,
                                bool pdl);
// Combines the partials of split blocks into attn16 (no launch when
// grid_chunks == 1).
cudaError_t launch_attn_merge(const PrefillAttnParams& p, cudaStream_t s, bool pdl);
cudaError_t configure_prefill_attn();

// Attention of a batched decode step (decode_batch.cu): B sequences, one new
// row each, caches [B][Hkv][max_ctx][D], slots [0, cache_lens[b]] (the last
// one already holding the new K/V).
struct DecodeAttnBatchParams {
  CUtensorMap tm_k;           // K cache viewed as (64, max_ctx, D / 64, B * Hkv), box
  CUtensorMap tm_v;           //   64 x 64 x D/64 x 1, SW128; the same for V (slots past
                              //   max_ctx read as zeros)
  const __half* q16;          // [B, Hq, D] (RoPE applied)
  const int64_t* cache_lens;  // [B], device
  int B, Hq, Hkv, D;
  int64_t max_ctx;
  float scale_log2;
  int64_t window;             // sliding window in slots (0 = full)
  int nsplit;                 // splits of each sequence's slots (decode_batch_splits)
  int deep;                   // decode_batch_deep: one CTA per SM of 8 warps
  float* part;                // [B][Hq][nsplit][D + 2] when nsplit > 1
  __half* attn16;             // [B, Hq * D]
  int* err;
  // K-split QKV (qkv_part != null, qkv_splits <= 4): the GEMM left qkv_splits fp32 partials
  // [S][B][(Hq + 2 Hkv) D]; this kernel adds them in split order, adds the
  // bias, rotates q and k at pos[b] and, in the CTA whose split holds slot
  // cache_lens[b], writes the new K/V there (and to k_new / v_new) before
  // reading it -- the work of qkv_finish, which is then not launched.  q16
  // is not used.
  const float* qkv_part;
  int qkv_splits;
  const __half* bias[3];      // q, k, v biases (null: none)
  const int64_t* pos;         // [B]
  const float2* rope;         // [rope_len][D / 2]
  int64_t rope_len;
  __half* kc;                 // caches [B][Hkv][max_ctx][D]
  __half* vc;
  __half* k_new;              // [B, Hkv, D] or null
  __half* v_new;
};
bool decode_batch_deep(int B, int Hkv, int num_sms);
int decode_batch_splits(int B, int Hkv, int64_t max_len, int num_sms);
size_t decode_batch_part_bytes(int B, int Hq, int D, int nsplit);
cudaError_t launch_decode_attn_batch(const DecodeAttnBatchParams& p, cudaStream_t s);
cudaError_t configure_decode_attn_batch();

// Final RMSNorm + LM head + greedy argmax (lm_head.cu).
struct LmHeadParams {
  CUtensorMap tm_w;     // W [vocab, H] viewed as (64, vocab, H / 64), box (64, 16, 24), SW128
  const __half* x;      // [T, H] last hidden rows (16-byte aligned)
  const __half* g;      // [H] final RMSNorm gain
  float eps;
  int T, H;             // 1 <= T <= 8, H % 64 == 0, H <= 4096
  int64_t vocab;
  float* logits;        // [T, vocab] fp32, may be null
  float* part_v;        // [num_sms][8] per-CTA best logit (workspace)
  int* part_i;          // [num_sms][8] its index
  int nparts;           // set by launch_lm_head
  int64_t* token;       // [T]
  int* err;
};
size_t lm_head_workspace_bytes(int num_sms);
cudaError_t launch_lm_head(LmHeadParams& p, int num_sms, cudaStream_t s, bool pdl);
cudaError_t launch_argmax_reduce(const LmHeadParams& p, cudaStream_t s);
cudaError_t launch_embed(const __half* table, int64_t vocab, const int64_t* ids, int T, int H,
                         __half* x, int* err, cudaStream_t s, bool pdl);
cudaError_t configure_lm_head();

// Sets the per-kernel shared-memory limits (called once per device).
// Quantized weights formed as fp16: fmt 1 INT8 (q int8 [rows, K], scale
// fp16 [rows]), fmt 2 int4 (packed uint8 [rows, K / 2], scale fp16 and zero
// uint8 [rows, K / group]); w fp16 [rows, K].  K a multiple of 16.
cudaError_t launch_dequant(int fmt, const void* q, const void* scale, const void* zero,
                           int64_t rows, int64_t K, int group, __half* w, int num_sms,
                           cudaStream_t s);

cudaError_t configure_kernels();

}  // namespace blk
