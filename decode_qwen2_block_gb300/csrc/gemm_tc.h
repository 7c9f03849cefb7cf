// tcgen05 GEMM for the prefill projections (see gemm_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace blk {

enum TcEpi {
  kTcQKV = 0,          // + bias, RoPE, q -> q16, k/v -> cache + k_new/v_new
  kTcResidF32 = 1,     // out32 = acc + res16         (o_proj)
  kTcGateUp = 2,       // out16 = silu(gate) * up     (B = W_gate | W_up)
  kTcResidOutF16 = 3   // out16 = acc + res32         (down)
};

struct TcGemmParams {
  CUtensorMap tmA;      // activations [M, K], box 64 x a_rows
  int a_rows;           // rows of tmA's box: 128, or M rounded up to 8 when M < 128
                        // (0 means 128); an M tile past M is not loaded at all
  CUtensorMap tmB[3];   // weights: QKV q/k/v; GATEUP gate/up; else [0]
  int M, N, K;          // N: output columns (QKV: (Hq+2Hkv)*D; GATEUP: I)
  int seg_rows[3];      // QKV: rows of wq, wk, wv
  int tiles_m, tiles_n, num_tiles;  // set by the launcher
  // QKV epilogue
  const __half* bias[3];
  const int64_t* pos;
  const float2* rope;
  int64_t rope_len;
  int Hq, Hkv, D;
  __half* q16;          // [M, Hq, D]
  __half* kc;
  __half* vc;
  __half* k_new;
  __half* v_new;
  int64_t max_ctx, cache_len;
  // batched decode (cache_lens != null): row m is sequence m, whose K/V go to
  // slot cache_lens[m] of the caches at kc/vc + m * seq_stride
  const int64_t* cache_lens;
  int64_t seq_stride;
  // other epilogues
  const __half* res16;
  const float* res32;
  float* out32;
  __half* out16;
  int ldo;
  // split K (any epilogue but gate/up, when part is set and max_splits > 1):
  // partials [splits][M][N] fp32; splits (<= max_splits) is chosen by the
  // launcher and the partials are finished by launch_splitk_reduce (down),
  // launch_qkv_finish (QKV) or launch_rmsnorm_splitk (o_proj)
  int splits;
  int max_splits;       // the partial buffer holds this many
  float* part;
  int* err;
};

// Rows of the activation box for an M-row operand: all 128 of a tile, or M
// rounded up to 8 when the operand is one partial tile (the tile rows past it
// are never stored, so they need not be loaded).
inline int tc_a_box_rows(int64_t M) { return M >= 128 ? 128 : (int)((M + 7) & ~int64_t(7)); }

// 2-D tensor map over a row-major [rows, K] fp16 matrix, box 64 x box_rows,
// 128-byte swizzle, zero fill out of bounds.  Returns 0 on success.
int make_tmap_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                 int box_rows);
// 3-D fp16 tensor map with 128-byte swizzle and zero fill: dims innermost
// first, strides (bytes) of dims 1 and 2, box sizes.  Returns 0 on success.
int make_tmap_3d(CUtensorMap* map, const void* base, const int64_t* dims,
                 const int64_t* strides, const int* box);
// The same with four dims (strides of dims 1..3 in bytes).
int make_tmap_4d(CUtensorMap* map, const void* base, const int64_t* dims,
                 const int64_t* strides, const int* box);
// Tensor map of 8-row weight boxes with 128-byte swizzle for the decode
// kernel: the 3-D view (64, rows, K / 64) with box (64, 8, cbs) when
// K % 64 == 0 (*is3d = 1), else the 2-D view (K, rows) with box (64, 8).
int make_tmap_rows8(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int cbs,
                    int* is3d);
// The same for a matrix of quantized codes viewed as bytes [rows, row_bytes]
// (row_bytes a multiple of 16): 3-D (128, rows, row_bytes / 128) with box
// (128, 8, cbs) when row_bytes % 128 == 0, else 2-D with box (128, 8).
int make_tmap_codes(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                    int cbs, int* is3d);

cudaError_t launch_tc_gemm(TcGemmParams& p, int epi, int num_sms, cudaStream_t s,
                           bool pdl);
// After a down-projection launch with p.splits > 1: out16 = fp16(sum of the
// split partials + res32) (N a multiple of 4).
cudaError_t launch_splitk_reduce(const TcGemmParams& p, int num_sms, cudaStream_t s);
// After a QKV launch with p.splits > 1: sums the partials in split order and
// applies the QKV epilogue (bias, RoPE, q16 / cache slot / k_new, v_new).
// (Batched decode with at most 4 splits leaves this to its attention kernel.)
cudaError_t launch_qkv_finish(const TcGemmParams& p, cudaStream_t s);
cudaError_t configure_tc_gemm_kernels();

}  // namespace blk
