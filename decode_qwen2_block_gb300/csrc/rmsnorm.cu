// Prefill-phase row RMSNorm: y = fp16(x * rsqrt(mean(x^2) + eps) * g), one CTA
// per row; x is the block input (fp16) or the fp32 residual stream h.
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

}  // namespace blk
