// Prefill-phase building blocks: row RMSNorm, a CUDA-core tiled GEMM with the
// block's fused epilogues, and the RoPE + KV-append kernel that turns the
// projected q/k/v rows into rotated q and cache entries.
#include "common.cuh"
#include "kernels.h"

namespace blk {

// ------------------------------------------------------------------ RMSNorm
// One CTA per row: y = fp16(x * rsqrt(mean(x^2) + eps) * g).
template <typename T>
__global__ void __launch_bounds__(256)
    rmsnorm_rows_kernel(const T* __restrict__ x, const __half* __restrict__ g,
                        int H, float eps, __half* __restrict__ y) {
  __shared__ float red[8];
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x, tid = threadIdx.x;
  const T* xr = x + (size_t)row * H;
  float ss = 0.f;
  for (int i = tid; i < H; i += 256) {
    const float v = (float)xr[i];
    ss += v * v;
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)H + eps);
  for (int i = tid; i < H; i += 256)
    y[(size_t)row * H + i] = __float2half_rn((float)xr[i] * r * __half2float(g[i]));
}

static cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t s, bool pdl,
                                   cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

cudaError_t launch_rmsnorm_rows(const void* x, bool x_is_f32, const __half* g,
                                int rows, int H, float eps, __half* y,
                                cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(rows), dim3(256), 0, s, pdl, attr);
  if (x_is_f32)
    return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel<float>,
                              static_cast<const float*>(x), g, H, eps, y);
  return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel<__half>,
                            static_cast<const __half*>(x), g, H, eps, y);
}

// --------------------------------------------------------------- SIMT GEMM
// 64x64 output tile, K step 32, 256 threads with a 4x4 micro-tile each.
constexpr int BM = 64, BN = 64, BK = 32;

template <int EPI>
__global__ void __launch_bounds__(256)
    gemm_simt_kernel(const __grid_constant__ GemmParams p) {
  constexpr bool kDual = (EPI == kEpiSwiGLU);
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float B2s[kDual ? BK : 1][BN + 4];
  griddep_wait();
  griddep_launch();
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {}, acc2[4][4] = {};
  // loader mapping: 64 rows x 32 k = 256 threads x 8 elements
  const int lr = tid / 4, lk = (tid % 4) * 8;
  for (int k0 = 0; k0 < p.K; k0 += BK) {
    {
      float f[8];
      const int m = m0 + lr, k = k0 + lk;
      if (m < p.M && k < p.K) {
        h8_to_f32(*reinterpret_cast<const uint4*>(p.A + (size_t)m * p.K + k), f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) As[lk + i][lr] = f[i];
      const int n = n0 + lr;
      if (n < p.N && k < p.K) {
        h8_to_f32(*reinterpret_cast<const uint4*>(p.B + (size_t)n * p.K + k), f);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) Bs[lk + i][lr] = f[i];
      if constexpr (kDual) {
        if (n < p.N && k < p.K) {
          h8_to_f32(*reinterpret_cast<const uint4*>(p.B2 + (size_t)n * p.K + k), f);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) B2s[lk + i][lr] = f[i];
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
      if constexpr (kDual) {
#pragma unroll
        for (int j = 0; j < 4; ++j) b2[j] = B2s[kk][tx + 16 * j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if constexpr (kDual) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
      if (m >= p.M || n >= p.N) continue;
      const size_t o = (size_t)m * p.ldo + n;
      if constexpr (EPI == kEpiStoreF32) {
        p.outF32[o] = acc[i][j];
      } else if constexpr (EPI == kEpiResidF32) {
        p.outF32[o] = acc[i][j] + __half2float(p.resF16[o]);
      } else if constexpr (EPI == kEpiSwiGLU) {
        p.outF16[o] = __float2half_rn(silu(acc[i][j]) * acc2[i][j]);
      } else {
        p.outF16[o] = __float2half_rn(acc[i][j] + p.resF32[o]);
      }
    }
}

cudaError_t launch_gemm(const GemmParams& p, int epi, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((p.N + BN - 1) / BN, (p.M + BM - 1) / BM),
                                    dim3(256), 0, s, pdl, attr);
  switch (epi) {
    case kEpiStoreF32: return cudaLaunchKernelEx(&cfg, gemm_simt_kernel<kEpiStoreF32>, p);
    case kEpiResidF32: return cudaLaunchKernelEx(&cfg, gemm_simt_kernel<kEpiResidF32>, p);
    case kEpiSwiGLU: return cudaLaunchKernelEx(&cfg, gemm_simt_kernel<kEpiSwiGLU>, p);
    default: return cudaLaunchKernelEx(&cfg, gemm_simt_kernel<kEpiResidOutF16>, p);
  }
}

// --------------------------------------------------------- RoPE + append
// One thread per (row t, head, pair i): adds the bias, rotates q and k pairs
// (i, i + D/2) with the gathered fp32 (cos, sin), writes q as fp16 and K/V to
// cache slot cache_len + t and to k_new / v_new.
__global__ void __launch_bounds__(256)
    rope_append_kernel(const __grid_constant__ RopeAppendParams p) {
  griddep_wait();
  griddep_launch();
  const int half = p.D / 2;
  const int heads = p.Hq + 2 * p.Hkv;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)p.T * heads * half;
  if (idx >= total) return;
  const int i = (int)(idx % half);
  const int hd = (int)((idx / half) % heads);
  const int t = (int)(idx / ((int64_t)half * heads));
  const int ncol = heads * p.D;
  const float* row = p.qkv32 + (size_t)t * ncol + (size_t)hd * p.D;
  float lo = row[i], hi = row[i + half];
  const int64_t pos = p.pos[t];
  const int64_t slot = p.cache_len + t;
  if (hd < p.Hq) {
    if (p.bq) {
      lo += __half2float(p.bq[hd * p.D + i]);
      hi += __half2float(p.bq[hd * p.D + half + i]);
    }
    const float2 cs = rope_cs(p.rope, p.rope_len, half, pos, i, p.err);
    __half* q = p.q16 + ((size_t)t * p.Hq + hd) * p.D;
    q[i] = __float2half_rn(lo * cs.x - hi * cs.y);
    q[half + i] = __float2half_rn(hi * cs.x + lo * cs.y);
  } else if (hd < p.Hq + p.Hkv) {
    const int g = hd - p.Hq;
    if (p.bk) {
      lo += __half2float(p.bk[g * p.D + i]);
      hi += __half2float(p.bk[g * p.D + half + i]);
    }
    const float2 cs = rope_cs(p.rope, p.rope_len, half, pos, i, p.err);
    const __half a = __float2half_rn(lo * cs.x - hi * cs.y);
    const __half b = __float2half_rn(hi * cs.x + lo * cs.y);
    __half* dst = p.kc + ((size_t)g * p.max_ctx + slot) * p.D;
    dst[i] = a;
    dst[half + i] = b;
    if (p.k_new) {
      p.k_new[((size_t)t * p.Hkv + g) * p.D + i] = a;
      p.k_new[((size_t)t * p.Hkv + g) * p.D + half + i] = b;
    }
  } else {
    const int g = hd - p.Hq - p.Hkv;
    if (p.bv) {
      lo += __half2float(p.bv[g * p.D + i]);
      hi += __half2float(p.bv[g * p.D + half + i]);
    }
    const __half a = __float2half_rn(lo), b = __float2half_rn(hi);
    __half* dst = p.vc + ((size_t)g * p.max_ctx + slot) * p.D;
    dst[i] = a;
    dst[half + i] = b;
    if (p.v_new) {
      p.v_new[((size_t)t * p.Hkv + g) * p.D + i] = a;
      p.v_new[((size_t)t * p.Hkv + g) * p.D + half + i] = b;
    }
  }
}

cudaError_t launch_rope_append(const RopeAppendParams& p, cudaStream_t s, bool pdl) {
  const int64_t total = (int64_t)p.T * (p.Hq + 2 * p.Hkv) * (p.D / 2);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((unsigned)((total + 255) / 256)), dim3(256), 0,
                                    s, pdl, attr);
  return cudaLaunchKernelEx(&cfg, rope_append_kernel, p);
}

}  // namespace blk
