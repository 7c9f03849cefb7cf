// Row RMSNorm of the prefill and batched-decode chains: y = fp16(x *
// rsqrt(mean(x^2) + eps) * g); x is the block input (fp16), the fp32 residual
// stream h, or (after a K-split o_proj) the sum of its partials and the block
// input, which is also written out as h.
#include "common.cuh"
#include "kernels.h"

namespace blk {

// ------------------------------------------------------------------ RMSNorm
// One warp per row.  Each lane loads its share of the row in batches of up to
// kMaxVec 16-byte vectors with every load of a batch in flight (a 1.5K-wide
// row is one batch, i.e. one memory round trip); the first batch stays in
// registers for the output pass, later batches are re-read.
constexpr int kNormWarps = 8;
constexpr int kMaxVec = 12;

template <typename T>
__device__ __forceinline__ float sumsq16(const uint4& v) {
  if constexpr (sizeof(T) == 2) {
    float f[8];
    h8_to_f32(v, f);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) s += f[e] * f[e];
    return s;
  } else {
    const float4 f = *reinterpret_cast<const float4*>(&v);
    return f.x * f.x + f.y * f.y + f.z * f.z + f.w * f.w;
  }
}

// Writes the normalised elements of vector i (8 fp16 or 4 fp32 inputs).
template <typename T>
__device__ __forceinline__ void put16(const uint4& v, int i, float r, const __half* g,
                                      __half* yr) {
  if constexpr (sizeof(T) == 2) {
    float f[8], gf[8];
    h8_to_f32(v, f);
    h8_to_f32(__ldg(reinterpret_cast<const uint4*>(g) + i), gf);
    uint4 o;
    __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      oh[e] = __floats2half2_rn(f[2 * e] * r * gf[2 * e], f[2 * e + 1] * r * gf[2 * e + 1]);
    reinterpret_cast<uint4*>(yr)[i] = o;
  } else {
    const float4 f = *reinterpret_cast<const float4*>(&v);
    const uint2 graw = __ldg(reinterpret_cast<const uint2*>(g) + i);
    const float2 ga = __half22float2(*reinterpret_cast<const __half2*>(&graw.x));
    const float2 gb = __half22float2(*reinterpret_cast<const __half2*>(&graw.y));
    uint2 o;
    *reinterpret_cast<__half2*>(&o.x) = __floats2half2_rn(f.x * r * ga.x, f.y * r * ga.y);
    *reinterpret_cast<__half2*>(&o.y) = __floats2half2_rn(f.z * r * gb.x, f.w * r * gb.y);
    reinterpret_cast<uint2*>(yr)[i] = o;
  }
}

template <typename T>
__global__ void __launch_bounds__(kNormWarps * 32)
    rmsnorm_rows_kernel(const T* __restrict__ x, const __half* __restrict__ g, int rows, int H,
                        float eps, __half* __restrict__ y) {
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kNormWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int nv = H / (16 / (int)sizeof(T));
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * H);
  uint4 v[kMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxVec; ++k) {
    const int i = lane + 32 * k;
    v[k] = i < nv ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int k = 0; k < kMaxVec; ++k) ss += sumsq16<T>(v[k]);
  for (int base = 32 * kMaxVec; base < nv; base += 32 * kMaxVec) {   // long rows
    uint4 w[kMaxVec];
#pragma unroll
    for (int k = 0; k < kMaxVec; ++k) {
      const int i = base + lane + 32 * k;
      w[k] = i < nv ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kMaxVec; ++k) ss += sumsq16<T>(w[k]);
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)H + eps);
  __half* yr = y + (size_t)row * H;
#pragma unroll
  for (int k = 0; k < kMaxVec; ++k) {
    const int i = lane + 32 * k;
    if (i < nv) put16<T>(v[k], i, r, g, yr);
  }
  for (int i = 32 * kMaxVec + lane; i < nv; i += 32) put16<T>(__ldg(xr + i), i, r, g, yr);
}

// After a K-split o_proj: h = (sum of the split partials, split order) + res16
// is written to h32 (the residual of the down projection) and y = RMSNorm(h)
// * g.  One CTA per row, four columns per thread and step; every partial of a
// step is loaded before any is added, so a row costs one memory round trip
// per step rather than one per split.
constexpr int kSplitNormMaxS = 8;

__global__ void __launch_bounds__(1024)
    rmsnorm_splitk_kernel(const float* __restrict__ part, int S, const __half* __restrict__ res16,
                          float* __restrict__ h32, const __half* __restrict__ g, int rows, int H,
                          float eps, __half* __restrict__ y) {
  __shared__ float red[32];
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x;
  const size_t MN = (size_t)rows * H, r0 = (size_t)row * H;
  float ss = 0.f;
  for (int i = 4 * threadIdx.x; i < H; i += 4 * blockDim.x) {
    float4 q[kSplitNormMaxS];
#pragma unroll
    for (int s = 0; s < kSplitNormMaxS; ++s)
      if (s < S) q[s] = __ldcg(reinterpret_cast<const float4*>(part + s * MN + r0 + i));
    const uint2 rr = __ldg(reinterpret_cast<const uint2*>(res16 + r0 + i));
    float4 a = q[0];
#pragma unroll
    for (int s = 1; s < kSplitNormMaxS; ++s)
      if (s < S) { a.x += q[s].x; a.y += q[s].y; a.z += q[s].z; a.w += q[s].w; }
    const float2 ra = __half22float2(*reinterpret_cast<const __half2*>(&rr.x));
    const float2 rb = __half22float2(*reinterpret_cast<const __half2*>(&rr.y));
    a.x += ra.x; a.y += ra.y; a.z += rb.x; a.w += rb.y;
    *reinterpret_cast<float4*>(h32 + r0 + i) = a;
    ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
  }
  ss = warp_sum(ss);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    float v = lane < nw ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = rsqrtf(red[0] / (float)H + eps);
  for (int i = 4 * threadIdx.x; i < H; i += 4 * blockDim.x) {   // this thread's own h32 values
    const float4 a = *reinterpret_cast<const float4*>(h32 + r0 + i);
    put16<float>(*reinterpret_cast<const uint4*>(&a), i / 4, r, g, y + r0);
  }
}

// After a K-split down projection inside a layer stack: the layer's output
// out16 = fp16(sum of the split partials, split order, + res32) -- the
// values splitk_reduce_kernel writes -- and the next layer's RMSNorm of that
// output, y = fp16(out * rsqrt(mean(out^2) + eps) * g), in one launch.  One
// CTA per row; each thread owns 8-column vectors i = t, t + blockDim, ...
// The squares are added exactly as rmsnorm_rows_kernel adds them for a
// one-warp row (per vector in column order; lane l then adds the vectors l,
// l + 32, ... in that order; then the warp's butterfly), so y has the same
// bits as a separate reduction followed by rmsnorm_rows.
constexpr int kReduceNormMaxS = 16;
constexpr int kReduceNormThreads = 256;

// MAXS (>= S) sizes the partial registers: 4 or 8 for the usual split
// counts keeps several blocks resident per SM when there are many rows.
template <int MAXS>
__global__ void __launch_bounds__(kReduceNormThreads)
    splitk_reduce_norm_kernel(const float* __restrict__ part, int S,
                              const float* __restrict__ res32, __half* __restrict__ out16,
                              const __half* __restrict__ g, int rows, int H, float eps,
                              __half* __restrict__ y) {
  extern __shared__ float vec_ss[];   // [H / 8] per-vector sums of squares
  __shared__ float r_row;
  griddep_wait();
  griddep_launch();
  const int row = blockIdx.x;
  const int nv = H / 8;
  const size_t MN = (size_t)rows * H, r0 = (size_t)row * H;
  uint4 first = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const size_t c = r0 + (size_t)i * 8;
    float4 q[MAXS][2];
#pragma unroll
    for (int j = 0; j < MAXS; ++j)
      if (j < S) {
        q[j][0] = __ldcg(reinterpret_cast<const float4*>(part + j * MN + c));
        q[j][1] = __ldcg(reinterpret_cast<const float4*>(part + j * MN + c) + 1);
      }
    const float4 ra = __ldcg(reinterpret_cast<const float4*>(res32 + c));
    const float4 rb = __ldcg(reinterpret_cast<const float4*>(res32 + c) + 1);
    float4 a = q[0][0], b = q[0][1];
#pragma unroll
    for (int j = 1; j < MAXS; ++j)
      if (j < S) {
        a.x += q[j][0].x; a.y += q[j][0].y; a.z += q[j][0].z; a.w += q[j][0].w;
        b.x += q[j][1].x; b.y += q[j][1].y; b.z += q[j][1].z; b.w += q[j][1].w;
      }
    uint4 o;
    *reinterpret_cast<__half2*>(&o.x) = __floats2half2_rn(a.x + ra.x, a.y + ra.y);
    *reinterpret_cast<__half2*>(&o.y) = __floats2half2_rn(a.z + ra.z, a.w + ra.w);
    *reinterpret_cast<__half2*>(&o.z) = __floats2half2_rn(b.x + rb.x, b.y + rb.y);
    *reinterpret_cast<__half2*>(&o.w) = __floats2half2_rn(b.z + rb.z, b.w + rb.w);
    reinterpret_cast<uint4*>(out16 + r0)[i] = o;
    vec_ss[i] = sumsq16<__half>(o);
    if (i == threadIdx.x) first = o;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < nv; i += 32) ss += vec_ss[i];
    ss = warp_sum(ss);
    if (threadIdx.x == 0) r_row = rsqrtf(ss / (float)H + eps);
  }
  __syncthreads();
  const float r = r_row;
  __half* yr = y + r0;
  for (int i = threadIdx.x; i < nv; i += blockDim.x)   // this thread's own output vectors
    put16<__half>(i == threadIdx.x ? first : reinterpret_cast<const uint4*>(out16 + r0)[i], i,
                  r, g, yr);
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
  cudaLaunchConfig_t cfg = make_cfg(dim3((rows + kNormWarps - 1) / kNormWarps),
                                    dim3(kNormWarps * 32), 0, s, pdl, attr);
  if (x_is_f32)
    return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel<float>,
                              static_cast<const float*>(x), g, rows, H, eps, y);
  return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel<__half>,
                            static_cast<const __half*>(x), g, rows, H, eps, y);
}

cudaError_t launch_rmsnorm_splitk(const float* part, int S, const __half* res16, float* h32,
                                  const __half* g, int rows, int H, float eps, __half* y,
                                  cudaStream_t s, bool pdl) {
  if (S < 1 || S > kSplitNormMaxS || H % 4) return cudaErrorInvalidValue;
  int threads = (H / 4 + 31) / 32 * 32;
  if (threads > 1024) threads = 1024;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(rows), dim3(threads), 0, s, pdl, attr);
  return cudaLaunchKernelEx(&cfg, rmsnorm_splitk_kernel, part, S, res16, h32, g, rows, H, eps,
                            y);
}

cudaError_t launch_splitk_reduce_norm(const float* part, int S, const float* res32,
                                      __half* out16, const __half* g, int rows, int H, float eps,
                                      __half* y, cudaStream_t s) {
  if (S < 1 || S > kReduceNormMaxS || H % 8) return cudaErrorInvalidValue;
  int threads = (H / 8 + 31) / 32 * 32;
  if (threads > kReduceNormThreads) threads = kReduceNormThreads;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(rows), dim3(threads), (size_t)(H / 8) * sizeof(float),
                                    s, true, attr);
  if (S <= 4)
    return cudaLaunchKernelEx(&cfg, splitk_reduce_norm_kernel<4>, part, S, res32, out16, g, rows,
                              H, eps, y);
  if (S <= 8)
    return cudaLaunchKernelEx(&cfg, splitk_reduce_norm_kernel<8>, part, S, res32, out16, g, rows,
                              H, eps, y);
  return cudaLaunchKernelEx(&cfg, splitk_reduce_norm_kernel<16>, part, S, res32, out16, g, rows,
                            H, eps, y);
}

}  // namespace blk
