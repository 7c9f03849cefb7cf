// Few-row projections of batched decode on the tensor cores (see gemm_fr.cu).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace blk {

constexpr int kFrMaxRows = 128;   // activation rows (sequences) the kernel takes

enum FrEpi {
  kFrPart = 0,     // fp32 partial of each K split: part[split][M][N]
  kFrGateUp = 1    // out16 = fp16(silu(x W_gate^T) * (x W_up^T)), no K split
};

struct FrGemmParams {
  // caller
  const void* x;          // activations [M, K] fp16, row-major, 16-byte aligned rows
  const void* w[3];       // weights [rows, K] fp16 (nn.Linear layout).  PART: up to
                          // three matrices stacked along N (QKV: wq, wk, wv), each
                          // seg_rows[i] rows, a multiple of 64 except the last;
                          // GATEUP: W_gate, W_up, both N rows
  int seg_rows[3];
  int M, N, K;            // M <= kFrMaxRows; N output columns; K % 8 == 0
  int max_splits;         // PART: the partial buffer holds this many splits
  float* part;            // PART: [splits][M][N] fp32
  __half* out16;          // GATEUP: [M][ldo] fp16
  int ldo;
  int* err;               // device status word (bounded-wait timeouts)
  // set by the launcher
  CUtensorMap tmX;        // box 64 x npad rows (rows past M read as zeros)
  CUtensorMap tmW[3];     // box 64 x 64 rows
  int npad;               // the MMA's N: M rounded up to 32, 64 or 128
  int splits;             // PART: K splits used (1 .. max_splits)
};

// Builds the tensor maps, picks the K split (PART: the largest that keeps
// every (tile, split) unit in one wave on num_sms SMs, at most max_splits and
// at most one per 64-column K block) and launches one CTA per unit.  Returns
// cudaErrorInvalidValue for a shape outside the limits above.
cudaError_t launch_fr_gemm(FrGemmParams& p, int epi, int num_sms, cudaStream_t s, bool pdl);
cudaError_t configure_fr_gemm_kernels();

}  // namespace blk
