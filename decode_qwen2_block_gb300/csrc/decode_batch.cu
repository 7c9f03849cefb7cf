// Attention of a batched decode step: B sequences, one new token each, every
// sequence with its own K/V cache and cache length (the decode phase of the
// TopOp decoder block, §4 "three-phase split": the new row attends to slots
// [0, cache_len] of its own cache, slot cache_len holding its new K/V).
//
// Split-K flash decode: CTA = (split, kv head g, sequence b), 4 warps.  The
// split's slots stream through a ring of 64-slot K/V tiles in shared memory
// (128-bit cp.async copies, 128-byte XOR swizzle, zero fill past the range).
// Two forms: when the (sequence, kv head) pairs are at most one per SM, one
// CTA per SM with a five-stage ring (four tiles in flight); otherwise two
// CTAs per SM with three stages.  The splits are chosen so that every CTA
// runs in one wave.
// Each warp owns 16 slots of a tile and runs mma.sync m16n8k16 with the G
// query heads of kv head g as the rows (padded to 16): S = Q K^T, an online
// base-2 softmax per head, O += P V; the warps' states are merged pairwise in
// shared memory.  One split writes attn directly; several write fp32
// partials (O, m, l) that decode_attn_merge_kernel combines in split order.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {
namespace {

constexpr int kTileSlots = 64;
constexpr int kStagesDeep = 5;             // one CTA per SM
constexpr int kStagesPair = 3;             // two CTAs per SM (at D = 128)
constexpr int kAWarps = 4;                 // 16 slots of a tile each
constexpr int kAThreads = kAWarps * 32;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
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

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 16-byte chunk `ch` (8 halves) of slot row r in a 64-slot tile stored as
// [D/64][64 rows][128 B] with the chunk index XORed by (r & 7).
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int ch) {
  return base + (ch >> 3) * (kTileSlots * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

// 16 bytes global -> shared; zeros instead when !valid (nothing is read).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D, int kStages>
struct BSmem {
  static constexpr int kQStride = D + 8;                      // halves (conflict-free ldmatrix)
  static constexpr int kTile = kTileSlots * D * 2;            // K or V tile bytes
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 16 * kQStride * 2;            // multiple of 16... rounded below
  static constexpr int kKVBase = (kKVOff + 1023) / 1024 * 1024;
  static constexpr int kOS = D + 8;                           // merge buffer row stride (floats)
  static constexpr int kBuf = 32 + 16 * kOS;                  // floats: m[16], l[16], o[16][kOS]
  static constexpr int kRing = kStages * 2 * kTile;           // (K, V) per stage
  // the warps' merge buffers reuse the ring once every tile has been used
  static constexpr int kMergeOff = kKVBase;
  static constexpr int kBody = kRing > 2 * kBuf * 4 ? kRing : 2 * kBuf * 4;
  static constexpr size_t kBytes = (size_t)kKVBase + kBody + 1024;
};

template <int D, int kStages>
__global__ void __launch_bounds__(kAThreads)
    decode_attn_batch_kernel(const __grid_constant__ DecodeAttnBatchParams p) {
  using Sm = BSmem<D, kStages>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __half* qtile = reinterpret_cast<__half*>(smem + Sm::kQOff);
  float* bufs = reinterpret_cast<float*>(smem + Sm::kMergeOff);
  const uint32_t kv0 = smem_u32(smem + Sm::kKVBase);

  griddep_wait();    // q, the caches' new slots and cache_lens come from earlier kernels
  griddep_launch();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = p.Hq / p.Hkv;
  const int64_t L = p.cache_lens[b];
  const int64_t n = (L >= 0 && L < p.max_ctx) ? L + 1 : 0;   // slots [0, L]
  const int64_t j0 = (int64_t)sp * n / p.nsplit, j1 = (int64_t)(sp + 1) * n / p.nsplit;
  const int ntiles = (int)((j1 - j0 + kTileSlots - 1) / kTileSlots);
  const size_t head = ((size_t)b * p.Hkv + g) * (size_t)p.max_ctx;
  const __half* kc = p.kc + head * D;
  const __half* vc = p.vc + head * D;
  constexpr int kCPR = D / 8;   // 16-byte chunks per row

  // Q tile: rows 0..G-1 = query heads g*G.., rows G..15 zero
  for (int i = tid; i < 16 * kCPR; i += kAThreads) {
    const int r = i / kCPR, ch = i % kCPR;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < G) v = *reinterpret_cast<const uint4*>(p.q16 + ((size_t)b * p.Hq + g * G + r) * D + ch * 8);
    *reinterpret_cast<uint4*>(qtile + r * Sm::kQStride + ch * 8) = v;
  }
  auto load_tile = [&](int t) {   // tile t into stage t % kStages (one copy group)
    const uint32_t kb = kv0 + (t % kStages) * 2 * Sm::kTile, vb = kb + Sm::kTile;
    const int64_t cs = j0 + (int64_t)t * kTileSlots;
    for (int i = tid; i < kTileSlots * kCPR; i += kAThreads) {
      const int r = i / kCPR, ch = i % kCPR;
      const int64_t j = cs + r;
      const bool valid = j < j1;
      const size_t off = (size_t)(valid ? j : j0) * D + ch * 8;
      cp_async16(tile_addr(kb, r, ch), kc + off, valid);
      cp_async16(tile_addr(vb, r, ch), vc + off, valid);
    }
    cp_async_commit();
  };
  // tiles 0 .. kStages-2 in flight; an empty group stands for a missing tile
  // so that "tile t has landed" is always "all but the newest kStages-2
  // groups have completed"
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) load_tile(s);
    else cp_async_commit();
  }

  const int grp = lane >> 2, tig = lane & 3;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float O[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
  const uint32_t qbase = smem_u32(qtile);
  const float sl2 = p.scale_log2;

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<kStages - 2>();   // tile t has landed (this thread's copies)
    __syncthreads();                // everyone's copies; stage (t-1) % kStages is free
    if (t + kStages - 1 < ntiles) load_tile(t + kStages - 1);
    else cp_async_commit();
    const uint32_t kb = kv0 + (t % kStages) * 2 * Sm::kTile, vb = kb + Sm::kTile;
    const int64_t cs = j0 + (int64_t)t * kTileSlots;
    const int nval = (int)min((int64_t)kTileSlots, j1 - cs);
    const int r0 = warp * 16;
    if (r0 < nval) {
      // S = Q K^T for this warp's 16 slots (two n-tiles of 8)
      float S[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4], bk[4];
        {
          const int m = lane >> 3, rr = (m & 1) * 8 + (lane & 7);
          const int col = ks * 16 + (m >> 1) * 8;
          ldsm_x4(qbase + (rr * Sm::kQStride + col) * 2, a);
        }
        {
          const int m = lane >> 3;
          const int r = r0 + (m >> 1) * 8 + (lane & 7);
          ldsm_x4(tile_addr(kb, r, ks * 2 + (m & 1)), bk);
        }
        mma16816(S[0], a, bk[0], bk[1]);
        mma16816(S[1], a, bk[2], bk[3]);
      }
      // online softmax in base 2 (rows grp and grp + 8 = query heads)
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = r0 + nt * 8 + 2 * tig + (e & 1);
          S[nt][e] = r >= nval ? -INFINITY : S[nt][e] * sl2;
          mx[e >> 1] = fmaxf(mx[e >> 1], S[nt][e]);
        }
      float corr[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
        mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
        const float mn = fmaxf(m_r[h2], mx[h2]);
        corr[h2] = (mn == -INFINITY) ? 1.f : exp2f(m_r[h2] - mn);
        m_r[h2] = mn;
        l_r[h2] *= corr[h2];
      }
      uint32_t pa[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mn = m_r[e >> 1];
          pv[e] = (S[nt][e] == -INFINITY || mn == -INFINITY) ? 0.f : exp2f(S[nt][e] - mn);
          l_r[e >> 1] += pv[e];
        }
        pa[2 * nt] = pack_h2(pv[0], pv[1]);
        pa[2 * nt + 1] = pack_h2(pv[2], pv[3]);
      }
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        O[dn][0] *= corr[0];
        O[dn][1] *= corr[0];
        O[dn][2] *= corr[1];
        O[dn][3] *= corr[1];
      }
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {   // O += P V
        uint32_t bv[4];
        const int m = lane >> 3;
        const int r = r0 + (m & 1) * 8 + (lane & 7);
        ldsm_x4_t(tile_addr(vb, r, dp * 2 + (m >> 1)), bv);
        mma16816(O[2 * dp], pa, bv[0], bv[1]);
        mma16816(O[2 * dp + 1], pa, bv[2], bv[3]);
      }
    }
  }
  cp_async_wait<0>();   // only empty groups can remain
  __syncthreads();      // every warp is done with the ring: the merge buffers reuse it

  // merge the warps' states: 1 -> 0, 3 -> 2, then 2 -> 0
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    l_r[h2] += __shfl_xor_sync(0xffffffffu, l_r[h2], 1);
    l_r[h2] += __shfl_xor_sync(0xffffffffu, l_r[h2], 2);
  }
  constexpr int kOS = Sm::kOS, kBuf = Sm::kBuf;
  auto put = [&](float* bf) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int row = grp + 8 * h2;
      if (tig == 0) {
        bf[row] = m_r[h2];
        bf[16 + row] = l_r[h2];
      }
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn)
        *reinterpret_cast<float2*>(bf + 32 + row * kOS + dn * 8 + 2 * tig) =
            make_float2(O[dn][2 * h2], O[dn][2 * h2 + 1]);
    }
  };
  auto merge_from = [&](const float* bf) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int row = grp + 8 * h2;
      const float mo = bf[row], lo = bf[16 + row];
      const float Mx = fmaxf(mo, m_r[h2]);
      const float a = (Mx == -INFINITY) ? 0.f : exp2f(mo - Mx);
      const float bs = (Mx == -INFINITY) ? 0.f : exp2f(m_r[h2] - Mx);
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const float2 o = *reinterpret_cast<const float2*>(bf + 32 + row * kOS + dn * 8 + 2 * tig);
        O[dn][2 * h2] = O[dn][2 * h2] * bs + o.x * a;
        O[dn][2 * h2 + 1] = O[dn][2 * h2 + 1] * bs + o.y * a;
      }
      l_r[h2] = l_r[h2] * bs + lo * a;
      m_r[h2] = Mx;
    }
  };
  if (warp & 1) put(bufs + (warp >> 1) * kBuf);
  __syncthreads();
  if (!(warp & 1)) merge_from(bufs + (warp >> 1) * kBuf);
  __syncthreads();
  if (warp == 2) put(bufs + kBuf);
  __syncthreads();
  if (warp == 0) {
    merge_from(bufs + kBuf);
    put(bufs);
  }
  __syncthreads();

  // rows < G: attn (one split) or this split's fp32 partial
  for (int i = tid; i < G * D; i += kAThreads) {
    const int row = i / D, d = i % D;
    const float m = bufs[row], l = bufs[16 + row], o = bufs[32 + row * kOS + d];
    const size_t bh = (size_t)b * p.Hq + g * G + row;
    if (p.nsplit == 1) {
      p.attn16[bh * D + d] = __float2half_rn(l > 0.f ? o / l : 0.f);
    } else {
      float* dst = p.part + (bh * p.nsplit + sp) * (size_t)(D + 2);
      dst[d] = o;
      if (d == 0) {
        dst[D] = m;
        dst[D + 1] = l;
      }
    }
  }
}

// attn[b, hq] = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, splits in order.
template <int D>
__global__ void __launch_bounds__(D) decode_attn_merge_kernel(const float* part, int nsplit,
                                                              __half* attn16) {
  griddep_wait();
  griddep_launch();
  const size_t bh = blockIdx.x;
  const int d = threadIdx.x;
  const float* P = part + bh * nsplit * (size_t)(D + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, P[s * (D + 2) + D]);
  float lt = 0.f, o = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = P[s * (D + 2) + D];
    const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
    lt = __fmaf_rn(w, P[s * (D + 2) + D + 1], lt);
    o = __fmaf_rn(w, P[s * (D + 2) + d], o);
  }
  attn16[bh * D + d] = __float2half_rn(lt > 0.f ? o / lt : 0.f);
}

}  // namespace

bool decode_batch_deep(int B, int Hkv, int num_sms) { return (int64_t)B * Hkv <= num_sms; }

// As many splits as keep every CTA in one wave (one CTA per SM in the deep
// form, two otherwise); at least one, at most one per 64-slot tile of the
// longest sequence.
int decode_batch_splits(int B, int Hkv, int64_t max_len, int num_sms) {
  const int64_t tiles = (max_len + 1 + kTileSlots - 1) / kTileSlots;
  const int per_sm = decode_batch_deep(B, Hkv, num_sms) ? 1 : 2;
  int64_t s = (int64_t)per_sm * num_sms / ((int64_t)B * Hkv);
  if (s > tiles) s = tiles;
  if (s > 256) s = 256;
  return (int)(s < 1 ? 1 : s);
}

size_t decode_batch_part_bytes(int B, int Hq, int D, int nsplit) {
  return nsplit > 1 ? (size_t)B * Hq * nsplit * (D + 2) * 4 : 0;
}

template <int D, int kStages>
static cudaError_t launch_attn_batch_d(const DecodeAttnBatchParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nsplit, p.Hkv, p.B);
  cfg.blockDim = dim3(kAThreads);
  cfg.dynamicSmemBytes = BSmem<D, kStages>::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_attn_batch_kernel<D, kStages>, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  cudaLaunchConfig_t mc = {};
  mc.gridDim = dim3(p.B * p.Hq);
  mc.blockDim = dim3(D);
  mc.stream = s;
  mc.attrs = attr;
  mc.numAttrs = 1;
  return cudaLaunchKernelEx(&mc, decode_attn_merge_kernel<D>, (const float*)p.part, p.nsplit,
                            p.attn16);
}

cudaError_t launch_decode_attn_batch(const DecodeAttnBatchParams& p, cudaStream_t s) {
  if (p.nsplit > 1 && !p.part) return cudaErrorInvalidValue;
  if (p.Hq / p.Hkv > 16) return cudaErrorInvalidValue;   // the rows of one MMA tile
  if (p.D == 128)
    return p.deep ? launch_attn_batch_d<128, kStagesDeep>(p, s)
                  : launch_attn_batch_d<128, kStagesPair>(p, s);
  if (p.D == 64)
    return p.deep ? launch_attn_batch_d<64, kStagesDeep>(p, s)
                  : launch_attn_batch_d<64, kStagesPair>(p, s);
  return cudaErrorInvalidValue;
}

template <int D, int kStages>
static cudaError_t configure_one() {
  return cudaFuncSetAttribute(decode_attn_batch_kernel<D, kStages>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)BSmem<D, kStages>::kBytes);
}

cudaError_t configure_decode_attn_batch() {
  cudaError_t e = configure_one<128, kStagesDeep>();
  if (e == cudaSuccess) e = configure_one<128, kStagesPair>();
  if (e == cudaSuccess) e = configure_one<64, kStagesDeep>();
  if (e == cudaSuccess) e = configure_one<64, kStagesPair>();
  return e;
}

}  // namespace blk
