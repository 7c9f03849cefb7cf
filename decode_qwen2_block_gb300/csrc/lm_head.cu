// Around the block stack: token embedding, and final RMSNorm + LM head +
// greedy argmax (the inference flow of the MLIR-compilation page, §2.3
// "LLM inference overview": embedding -> blocks -> LM head -> logits ->
// sampling; greedy argmax over the vocabulary as in the buddy-mlir
// DeepSeek-R1 page, §6.4.4 and §6.4.6).
//
// The LM head is a matrix-vector product over vocab x H fp16 weights (467 MB
// for 151936 x 1536): it is bound by HBM bytes.  lm_head_kernel runs one CTA
// per SM; each streams a contiguous range of 16-row weight groups through a
// four-stage (hidden <= 2048; else three-stage) shared-memory ring (one 3-D
// TMA copy of 16 rows x 1536 columns, 48 KB, 128-byte swizzle, per stage)
// while one consumer warp per stage multiplies them on the tensor cores (mma.sync m16n8k16: A = 16 weight
// rows x 16 columns by ldmatrix, B = the T <= 8 normalised hidden rows, fp32
// accumulation).  The normalised rows y = RMSNorm(x) * g are computed by the
// consumer warps while the first copies are in flight (weights never depend
// on the token).  Each lane keeps the best (logit, index) of its token
// columns; the CTA's best per token goes to the workspace and
// argmax_reduce_kernel picks the largest logit, lowest index on ties.
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {
namespace {

constexpr int kGroupRows = 16;          // weight rows per group (MMA M)
constexpr int kCB = 24;                 // 64-column blocks per ring stage
constexpr int kChunkCols = kCB * 64;    // 1536
constexpr int kStageBytes = kGroupRows * kChunkCols * 2;   // 48 KB
constexpr int kMaxT = 8;                // MMA N
// NS consumer warps = ring stages; the normalised rows take the rest of
// shared memory: four stages for hidden <= 2048, three up to 4096.
template <int NS>
struct LmCfg {
  static constexpr int kThreads = (NS + 1) * 32;
  static constexpr int kMaxH = NS == 4 ? 2048 : 4096;
  static constexpr int kYStride = kMaxH + 8;   // halves; +16 B per row: conflict-free B loads
  static constexpr size_t kSmemBytes =
      (size_t)NS * kStageBytes + (size_t)kMaxT * kYStride * 2 + 256 + 1024;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (value, index) order of the argmax: larger value, then lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// The work of consumer warp w: groups first + w, first + w + NS, ... of the
// CTA's range [first, last), each in nck chunks of kChunkCols columns.
template <int NS>
struct WarpItems {
  int first, last, nck;
  __device__ int count(int w) const {
    const int groups = last - first - w;
    return groups <= 0 ? 0 : ((groups + NS - 1) / NS) * nck;
  }
  __device__ int group(int w, int n) const { return first + w + NS * (n / nck); }
};

template <int NS>
__global__ void __launch_bounds__(LmCfg<NS>::kThreads, 1)
    lm_head_kernel(const __grid_constant__ LmHeadParams p) {
  constexpr int kCWarps = NS;
  constexpr int kYStride = LmCfg<NS>::kYStride;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  __half* ys = reinterpret_cast<__half*>(smem + kCWarps * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kCWarps * kStageBytes +
                                               (size_t)kMaxT * kYStride * 2);
  uint64_t* full = bars;                 // [kCWarps]
  uint64_t* empty = bars + kCWarps;      // [kCWarps]
  float* best_v = reinterpret_cast<float*>(bars + 2 * kCWarps);   // [kCWarps][kMaxT]
  int* best_i = reinterpret_cast<int*>(best_v + kCWarps * kMaxT); // [kCWarps][kMaxT]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = (int)((p.vocab + kGroupRows - 1) / kGroupRows);
  WarpItems<NS> wi;
  wi.first = (int)((int64_t)blockIdx.x * ngroups / gridDim.x);
  wi.last = (int)((int64_t)(blockIdx.x + 1) * ngroups / gridDim.x);
  wi.nck = (p.H + kChunkCols - 1) / kChunkCols;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kCWarps; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCWarps) {
    // ------------------------------------------------------------ producer
    // The weights do not depend on the previous kernel: no dependency wait.
    if (lane == 0) {
      int cnt[kCWarps], issued[kCWarps];
      int most = 0;
      for (int w = 0; w < kCWarps; ++w) {
        cnt[w] = wi.count(w);
        issued[w] = 0;
        most = max(most, cnt[w]);
      }
      bool ok = true;
      for (int n = 0; n < most && ok; ++n) {
        for (int w = 0; w < kCWarps; ++w) {
          if (n >= cnt[w]) continue;
          if (n > 0 && !mbar_wait(&empty[w], (n - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[w], kStageBytes);
          tma_load_3d(smem_u32(ring + (size_t)w * kStageBytes), &p.tm_w, 0,
                      wi.group(w, n) * kGroupRows, (n % wi.nck) * kCB, &full[w]);
          ++issued[w];
        }
      }
      // copies in flight land before shared memory goes away
      for (int w = 0; w < kCWarps; ++w)
        if (issued[w] > 0) mbar_wait(&full[w], (issued[w] - 1) & 1, nullptr);
    }
  } else {
    // ------------------------------------------------------------ consumers
    griddep_wait();   // x comes from the previous kernel
    // y[t] = fp16(RMSNorm(x[t]) * g) for t < T, zero rows up to kMaxT
    for (int t = warp; t < kMaxT; t += kCWarps) {
      __half* yr = ys + t * kYStride;
      if (t >= p.T) {
        for (int i = lane * 8; i < p.H; i += 256) *reinterpret_cast<uint4*>(yr + i) = make_uint4(0, 0, 0, 0);
        continue;
      }
      const __half* xr = p.x + (size_t)t * p.H;
      float ss = 0.f;
      for (int i = lane * 8; i < p.H; i += 256) {
        float f[8];
        h8_to_f32(__ldg(reinterpret_cast<const uint4*>(xr + i)), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss += f[e] * f[e];
      }
      ss = warp_sum(ss);
      const float r = rsqrtf(ss / (float)p.H + p.eps);
      for (int i = lane * 8; i < p.H; i += 256) {
        float f[8];
        h8_to_f32(__ldg(reinterpret_cast<const uint4*>(xr + i)), f);
        uint4 o;
        __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          oh[e] = __floats2half2_rn(f[2 * e] * r * __half2float(p.g[i + 2 * e]),
                                    f[2 * e + 1] * r * __half2float(p.g[i + 2 * e + 1]));
        *reinterpret_cast<uint4*>(yr + i) = o;
      }
    }
    named_sync(1, kCWarps * 32);   // every consumer warp reaches this once

    const int gq = lane >> 2, tg = lane & 3;          // accumulator row / token pair
    const int m8 = lane >> 3, r16 = (lane & 7) + 8 * (m8 & 1), khalf = m8 >> 1;
    const uint32_t stage = smem_u32(ring + (size_t)warp * kStageBytes);
    const __half* yb = ys + gq * kYStride + 2 * tg;   // B: token gq, k pair 2tg
    float bv0 = -INFINITY, bv1 = -INFINITY;           // tokens 2tg and 2tg + 1
    int bi0 = 0x7fffffff, bi1 = 0x7fffffff;
    const int cnt = wi.count(warp);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    for (int n = 0; n < cnt; ++n) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[warp], n & 1, p.err))) {
        ok = false;
        break;
      }
      const int kc = n % wi.nck;
      const int nks = min(kChunkCols, p.H - kc * kChunkCols) / 16;
      const __half* yk = yb + kc * kChunkCols;
#pragma unroll 4
      for (int ks = 0; ks < nks; ++ks) {
        uint32_t a[4];
        // 16-byte chunk (ks % 4) * 2 + khalf of row r16 in column block ks / 4
        ldsm_x4(stage + (ks >> 2) * (kGroupRows * 128) + r16 * 128 +
                    (((((ks & 3) << 1) | khalf) ^ (r16 & 7)) << 4),
                a);
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(yk + ks * 16);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(yk + ks * 16 + 8);
        mma16816(d, a, b0, b1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[warp]);
      if (kc == wi.nck - 1) {   // the group is complete: rows g*16 + gq (+ 8)
        const int v0 = wi.group(warp, n) * kGroupRows + gq, v1 = v0 + 8;
        const int t0 = 2 * tg, t1 = t0 + 1;
        if (v0 < p.vocab) {
          if (t0 < p.T) {
            if (p.logits) p.logits[(size_t)t0 * p.vocab + v0] = d[0];
            if (better(d[0], v0, bv0, bi0)) { bv0 = d[0]; bi0 = v0; }
          }
          if (t1 < p.T) {
            if (p.logits) p.logits[(size_t)t1 * p.vocab + v0] = d[1];
            if (better(d[1], v0, bv1, bi1)) { bv1 = d[1]; bi1 = v0; }
          }
        }
        if (v1 < p.vocab) {
          if (t0 < p.T) {
            if (p.logits) p.logits[(size_t)t0 * p.vocab + v1] = d[2];
            if (better(d[2], v1, bv0, bi0)) { bv0 = d[2]; bi0 = v1; }
          }
          if (t1 < p.T) {
            if (p.logits) p.logits[(size_t)t1 * p.vocab + v1] = d[3];
            if (better(d[3], v1, bv1, bi1)) { bv1 = d[3]; bi1 = v1; }
          }
        }
        d[0] = d[1] = d[2] = d[3] = 0.f;
      }
    }
    // best over the lanes holding the same tokens (same tg), then over warps
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      const float ov0 = __shfl_xor_sync(0xffffffffu, bv0, off);
      const int oi0 = __shfl_xor_sync(0xffffffffu, bi0, off);
      const float ov1 = __shfl_xor_sync(0xffffffffu, bv1, off);
      const int oi1 = __shfl_xor_sync(0xffffffffu, bi1, off);
      if (better(ov0, oi0, bv0, bi0)) { bv0 = ov0; bi0 = oi0; }
      if (better(ov1, oi1, bv1, bi1)) { bv1 = ov1; bi1 = oi1; }
    }
    if (gq == 0) {
      best_v[warp * kMaxT + 2 * tg] = bv0;
      best_i[warp * kMaxT + 2 * tg] = bi0;
      best_v[warp * kMaxT + 2 * tg + 1] = bv1;
      best_i[warp * kMaxT + 2 * tg + 1] = bi1;
    }
    if (!ok) set_error(p.err, kDevTimeout);
    named_sync(1, kCWarps * 32);
    if (warp == 0 && lane < p.T) {
      float v = best_v[lane];
      int i = best_i[lane];
      for (int w = 1; w < kCWarps; ++w)
        if (better(best_v[w * kMaxT + lane], best_i[w * kMaxT + lane], v, i)) {
          v = best_v[w * kMaxT + lane];
          i = best_i[w * kMaxT + lane];
        }
      p.part_v[(size_t)blockIdx.x * kMaxT + lane] = v;
      p.part_i[(size_t)blockIdx.x * kMaxT + lane] = i;
    }
    griddep_launch();
  }
}

// token[t] = index of the best (value, index) over the CTAs' candidates.
__global__ void __launch_bounds__(kMaxT * 32) argmax_reduce_kernel(const float* part_v,
                                                                  const int* part_i, int nparts,
                                                                  int T, int64_t vocab,
                                                                  int64_t* token, int* err) {
  griddep_wait();
  const int t = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (t >= T) return;
  float v = -INFINITY;
  int i = 0x7fffffff;
  for (int b = lane; b < nparts; b += 32) {
    const float bv = part_v[(size_t)b * kMaxT + t];
    const int bi = part_i[(size_t)b * kMaxT + t];
    if (better(bv, bi, v, i)) { v = bv; i = bi; }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
  if (lane == 0) {
    if (i < 0 || i >= vocab) {   // no finite logit (NaN everywhere)
      set_error(err, kDevToken);
      i = 0;
    }
    token[t] = i;
  }
}

// x[t, :] = table[ids[t], :]; an id outside [0, vocab) records kDevToken and
// gives a zero row.
__global__ void __launch_bounds__(128) embed_kernel(const __half* table, int64_t vocab,
                                                    const int64_t* ids, int H, __half* x,
                                                    int* err) {
  griddep_wait();
  griddep_launch();
  const int t = blockIdx.x;
  const int64_t id = ids[t];
  const bool ok = id >= 0 && id < vocab;
  if (!ok && threadIdx.x == 0) set_error(err, kDevToken);
  const uint4* src = reinterpret_cast<const uint4*>(table + (ok ? id : 0) * (int64_t)H);
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)t * H);
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x)
    dst[i] = ok ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
}

}  // namespace

size_t lm_head_workspace_bytes(int num_sms) {
  return (size_t)num_sms * kMaxT * (sizeof(float) + sizeof(int));
}

template <int NS>
static cudaError_t launch_ns(LmHeadParams& p, int num_sms, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(LmCfg<NS>::kThreads);
  cfg.dynamicSmemBytes = LmCfg<NS>::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  p.nparts = num_sms;
  return cudaLaunchKernelEx(&cfg, lm_head_kernel<NS>, p);
}

cudaError_t launch_lm_head(LmHeadParams& p, int num_sms, cudaStream_t s, bool pdl) {
  if (p.T < 1 || p.T > kMaxT || p.H < 64 || p.H > LmCfg<3>::kMaxH || p.H % 64)
    return cudaErrorInvalidValue;
  return p.H <= LmCfg<4>::kMaxH ? launch_ns<4>(p, num_sms, s, pdl) : launch_ns<3>(p, num_sms, s, pdl);
}

cudaError_t launch_argmax_reduce(const LmHeadParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kMaxT * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, argmax_reduce_kernel, (const float*)p.part_v,
                            (const int*)p.part_i, p.nparts, p.T, p.vocab, p.token, p.err);
}

cudaError_t launch_embed(const __half* table, int64_t vocab, const int64_t* ids, int T, int H,
                         __half* x, int* err, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, embed_kernel, table, vocab, ids, H, x, err);
}

cudaError_t configure_lm_head() {
  const cudaError_t e = cudaFuncSetAttribute(lm_head_kernel<4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)LmCfg<4>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lm_head_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)LmCfg<3>::kSmemBytes);
}

}  // namespace blk
