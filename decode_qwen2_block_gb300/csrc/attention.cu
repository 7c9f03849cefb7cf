// Causal GQA attention over the fp16 KV cache for prefill / prefill_kv: one
// warp per (new row t, kv head g) over slots [0, cache_len + t], keeping for
// all G = Hq/Hkv query heads of the group the running max, sum and
// unnormalised output (online softmax, base-2 exponent with log2(e)/sqrt(D)
// folded into q).  Scores use one lane per slot (a full K row per lane, q
// broadcast from shared memory); the V accumulation uses lanes along D.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {

template <int G, int D>
struct WarpState {
  float m[G], l[G], acc[G][D / 32];
};

// Streams slots [j0, j1) of one kv head.  q_s: shared [G][D] fp32, already
// scaled by log2(e)/sqrt(D).  K, V point at slot 0 of the head (stride D).
template <int G, int D>
__device__ __forceinline__ void warp_attend(const float* q_s, const __half* K,
                                            const __half* V, int64_t j0,
                                            int64_t j1, WarpState<G, D>& st) {
  constexpr int DPL = D / 32;  // elements of D per lane in the V pass
  const int lane = threadIdx.x & 31;
  for (int64_t base = j0; base < j1; base += 32) {
    const int64_t j = base + lane;
    const bool valid = j < j1;
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) sc[h] = 0.f;
    if (valid) {
      const uint4* krow = reinterpret_cast<const uint4*>(K + j * D);
#pragma unroll 2
      for (int v = 0; v < D / 8; ++v) {
        float kf[8];
        h8_to_f32(__ldg(krow + v), kf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 qa = *reinterpret_cast<const float4*>(q_s + h * D + 8 * v);
          const float4 qb = *reinterpret_cast<const float4*>(q_s + h * D + 8 * v + 4);
          sc[h] += qa.x * kf[0] + qa.y * kf[1] + qa.z * kf[2] + qa.w * kf[3] +
                   qb.x * kf[4] + qb.y * kf[5] + qb.z * kf[6] + qb.w * kf[7];
        }
      }
    }
    float p[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float s = valid ? sc[h] : -INFINITY;
      const float mx = warp_max(s);
      const float m_new = fmaxf(st.m[h], mx);
      const float corr = exp2f(st.m[h] - m_new);  // 0 when m was -inf
      p[h] = valid ? exp2f(s - m_new) : 0.f;
      st.l[h] = st.l[h] * corr + warp_sum(p[h]);
      st.m[h] = m_new;
#pragma unroll
      for (int e = 0; e < DPL; ++e) st.acc[h][e] *= corr;
    }
    const int nvalid = (int)min((int64_t)32, j1 - base);
    for (int jj = 0; jj < nvalid; ++jj) {
      float vf[DPL];
      const __half* vrow = V + (base + jj) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(vrow));
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        vf[0] = a.x; vf[1] = a.y; vf[2] = b.x; vf[3] = b.y;
      } else {
        const float2 a = __half22float2(__ldg(reinterpret_cast<const __half2*>(vrow)));
        vf[0] = a.x; vf[1] = a.y;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pj = __shfl_sync(0xffffffffu, p[h], jj);
#pragma unroll
        for (int e = 0; e < DPL; ++e) st.acc[h][e] = fmaf(pj, vf[e], st.acc[h][e]);
      }
    }
  }
}

template <int G, int D>
__device__ __forceinline__ void init_state(WarpState<G, D>& st) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    st.m[h] = -INFINITY;
    st.l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) st.acc[h][e] = 0.f;
  }
}

template <int G, int D>
__global__ void __launch_bounds__(32)
    prefill_attn_simple_kernel(const __grid_constant__ PrefillAttnParams p) {
  __shared__ __align__(16) float q_s[G * D];
  const int t = blockIdx.x, g = blockIdx.y, lane = threadIdx.x;
  constexpr int DPL = D / 32;
  griddep_wait();
  griddep_launch();
  for (int i = lane; i < G * D; i += 32)
    q_s[i] = __half2float(p.q16[((size_t)t * p.Hq + g * G) * D + i]) * p.scale_log2;
  __syncwarp();
  WarpState<G, D> st;
  init_state(st);
  const size_t head_off = (size_t)g * p.max_ctx * D;
  warp_attend<G, D>(q_s, p.kc + head_off, p.vc + head_off, 0, p.cache_len + t + 1, st);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float inv = 1.f / st.l[h];
#pragma unroll
    for (int e = 0; e < DPL; ++e)
      p.attn16[(size_t)t * p.Hq * D + (g * G + h) * D + lane * DPL + e] =
          __float2half_rn(st.acc[h][e] * inv);
  }
}

// ---------------------------------------------------------------- host side

template <int G, int D>
static cudaError_t launch_pre(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.T, p.Hkv);
  cfg.blockDim = dim3(32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prefill_attn_simple_kernel<G, D>, p);
}

#define BLK_GD_DISPATCH(FN, P, S, PDL)                         \
  do {                                                         \
    const int G_ = (P).Hq / (P).Hkv;                           \
    if ((P).D == 128) {                                        \
      switch (G_) {                                            \
        case 1: return FN<1, 128>(P, S, PDL);                  \
        case 2: return FN<2, 128>(P, S, PDL);                  \
        case 4: return FN<4, 128>(P, S, PDL);                  \
        case 6: return FN<6, 128>(P, S, PDL);                  \
        case 8: return FN<8, 128>(P, S, PDL);                  \
        case 16: return FN<16, 128>(P, S, PDL);                \
      }                                                        \
    } else if ((P).D == 64) {                                  \
      switch (G_) {                                            \
        case 1: return FN<1, 64>(P, S, PDL);                   \
        case 2: return FN<2, 64>(P, S, PDL);                   \
        case 4: return FN<4, 64>(P, S, PDL);                   \
        case 6: return FN<6, 64>(P, S, PDL);                   \
        case 8: return FN<8, 64>(P, S, PDL);                   \
        case 16: return FN<16, 64>(P, S, PDL);                 \
      }                                                        \
    }                                                          \
    return cudaErrorInvalidValue;                              \
  } while (0)

cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  BLK_GD_DISPATCH(launch_pre, p, s, pdl);
}

}  // namespace blk
