// Attention of a batched decode step: B sequences, one new token each, every
// sequence with its own K/V cache and cache length (the decode phase of the
// TopOp decoder block, §4 "three-phase split": the new row attends to slots
// [0, cache_len] of its own cache, slot cache_len holding its new K/V).
//
// Split-K flash decode: CTA = (split, kv head g, sequence b), 4 warps.  The
// split's slots stream through a ring of 64-slot K/V tiles in shared memory
// (one TMA tensor copy per K or V tile, 128-byte swizzle, zero fill past
// max_ctx; rows past the split's end are masked).
// Two forms: when the (sequence, kv head) pairs are at most one per SM, one
// CTA per SM of 8 warps that use two tiles at a time, with three such pairs
// in the ring (four tiles in flight); otherwise two CTAs per SM of 4 warps
// with three tiles.  The splits are chosen so that every CTA runs in one wave.
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
// The ring holds kGroups copy groups of kTPG tiles; 4 * kTPG warps use one
// group at a time, four warps (16 slots each) per tile.
constexpr int kGroupsDeep = 3, kTpgDeep = 2;   // one CTA per SM, 8 warps
constexpr int kGroupsPair = 3, kTpgPair = 1;   // two CTAs per SM (at D = 128), 4 warps

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

// One box (0, y, 0, z) of a 4-D tensor map into shared memory; completion is
// counted on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(0), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// tensor (async-proxy) copies into the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The same for global memory: this thread's stores before later tensor
// copies that read them.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The attention kernel finishes a K-split QKV projection of at most this
// many splits (more: qkv_finish does it first).
constexpr int kQkvMaxSplits = 4;

// Column pair (c0, c0 + D/2) of row b of the K-split QKV output: the S
// partials (every load issued before any add), added in split order, plus
// the bias pair.
struct QkvPair {
  float a[kQkvMaxSplits], c[kQkvMaxSplits];
  float ba, bc;
};
__device__ __forceinline__ void qkv_pair_load(const DecodeAttnBatchParams& p, int b, int c0,
                                              int half, const __half* bias, int bi, QkvPair& q) {
  const size_t N = (size_t)(p.Hq + 2 * p.Hkv) * p.D, MN = (size_t)p.B * N;
  const float* src = p.qkv_part + (size_t)b * N + c0;
#pragma unroll
  for (int s = 0; s < kQkvMaxSplits; ++s)
    if (s < p.qkv_splits) {
      q.a[s] = __ldcg(src + s * MN);
      q.c[s] = __ldcg(src + s * MN + half);
    }
  q.ba = bias ? __half2float(bias[bi]) : 0.f;
  q.bc = bias ? __half2float(bias[bi + half]) : 0.f;
}
__device__ __forceinline__ float2 qkv_pair_sum(const DecodeAttnBatchParams& p, const QkvPair& q) {
  float a = 0.f, c = 0.f;
#pragma unroll
  for (int s = 0; s < kQkvMaxSplits; ++s)
    if (s < p.qkv_splits) {
      a += q.a[s];
      c += q.c[s];
    }
  return make_float2(a + q.ba, c + q.bc);
}

template <int D, int kGroups, int kTPG>
struct BSmem {
  static constexpr int kQStride = D + 8;                      // halves (conflict-free ldmatrix)
  static constexpr int kTile = kTileSlots * D * 2;            // K or V tile bytes
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 16 * kQStride * 2;            // multiple of 16... rounded below
  static constexpr int kKVBase = (kKVOff + 1023) / 1024 * 1024;
  static constexpr int kBarOff = kKVBase - 64;                // kGroups mbarriers
  static_assert(kKVOff <= kBarOff && kGroups <= 8, "barrier area");
  static constexpr int kOS = D + 8;                           // merge buffer row stride (floats)
  static constexpr int kBuf = 32 + 16 * kOS;                  // floats: m[16], l[16], o[16][kOS]
  static constexpr int kRing = kGroups * kTPG * 2 * kTile;   // (K, V) per tile
  // the warps' merge buffers (half the warps' states at once) reuse the
  // ring once every tile has been used
  static constexpr int kMergeOff = kKVBase;
  static constexpr int kMergeBytes = 2 * kTPG * kBuf * 4;
  static constexpr int kBody = kRing > kMergeBytes ? kRing : kMergeBytes;
  static constexpr size_t kBytes = (size_t)kKVBase + kBody + 1024;
};

template <int D, int kGroups, int kTPG>
__global__ void __launch_bounds__(128 * kTPG)
    decode_attn_batch_kernel(const __grid_constant__ DecodeAttnBatchParams p) {
  using Sm = BSmem<D, kGroups, kTPG>;
  constexpr int kWarps = 4 * kTPG, kThreads = 32 * kWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __half* qtile = reinterpret_cast<__half*>(smem + Sm::kQOff);
  float* bufs = reinterpret_cast<float*>(smem + Sm::kMergeOff);
  const uint32_t kv0 = smem_u32(smem + Sm::kKVBase);

  // Before griddepcontrol.wait only what the previous kernel of the chain
  // (qkv_finish) does not write may be read: everything older is complete
  // when this kernel starts, so the cache lengths and the history slots
  // below L are final; q and slot L are not.
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = p.Hq / p.Hkv;
  const int64_t L = p.cache_lens[b];
  const int64_t n = (L >= 0 && L < p.max_ctx) ? L + 1 : 0;   // slots [0, L]
  const int64_t lo = n > 0 ? window_lo(p.window, L) : 0;        // or the window's part
  const int64_t j0 = lo + (int64_t)sp * (n - lo) / p.nsplit;
  const int64_t j1 = lo + (int64_t)(sp + 1) * (n - lo) / p.nsplit;
  const int ntiles = (int)((j1 - j0 + kTileSlots - 1) / kTileSlots);
  const int ngroups = (ntiles + kTPG - 1) / kTPG;
  const int zh = b * p.Hkv + g;   // this (sequence, kv head) in the tensor maps
  constexpr int kCPR = D / 8;     // 16-byte chunks per row
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);   // [kGroups]
  // Tile slot u of the ring: K at kv0 + u * 2 * kTile, V right after it, each
  // [D/64][64 slots][128 B] with the 128-byte swizzle (the tensor copies' own
  // layout).  Thread 0 loads group gi (tiles gi*kTPG..) into ring group
  // gi % kGroups, completing on full[gi % kGroups].  Slots past the split's
  // end inside a tile are real cache rows (or zeros past max_ctx); they are
  // masked out below.
  auto group_nt = [&](int gi) { return min(kTPG, ntiles - gi * kTPG); };
  auto load_group = [&](int gi) {
    const int nt = group_nt(gi);
    uint64_t* bar = &full[gi % kGroups];
    fence_proxy_async_smem();   // the previous use of this group came first
    mbar_arrive_expect_tx(bar, (uint32_t)(nt * 2 * Sm::kTile));
    for (int jt = 0; jt < nt; ++jt) {
      const uint32_t kb = kv0 + ((gi % kGroups) * kTPG + jt) * 2 * Sm::kTile, vb = kb + Sm::kTile;
      const int y = (int)(j0 + (int64_t)(gi * kTPG + jt) * kTileSlots);
      tma_load_4d(kb, &p.tm_k, y, zh, bar);   // the tile's D/64 halves in one copy each
      tma_load_4d(vb, &p.tm_v, y, zh, bar);
    }
  };
  int issued = 0;   // thread 0: groups loaded so far
  if (tid == 0) {
    for (int s = 0; s < kGroups; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    // groups whose boxes end before slot L, ahead of the wait
    while (issued < kGroups - 1 && issued < ngroups &&
           j0 + (int64_t)(issued * kTPG + group_nt(issued)) * kTileSlots <= L)
      load_group(issued++);
  }
  griddep_wait();    // q and the new slot L come from the previous kernel
  griddep_launch();

  if (p.qkv_part) {
    // the QKV projection's K splits: q of this CTA's G heads (rows G..15
    // zero), and in the split that holds slot L the new K/V, stored in the
    // cache before the copies below read that slot
    constexpr int half = D / 2;
    const int64_t ps = p.pos[b];
    const bool pos_ok = ps >= 0 && ps < p.rope_len;
    if (!pos_ok && tid == 0 && sp == 0 && g == 0) set_error(p.err, kDevPosition);
    const float2* cs = p.rope + (size_t)(pos_ok ? ps : 0) * half;
    // every thread's loads of every item first (one round trip), then the
    // sums; rows G..15 of the tile are zero
    constexpr int kItems = (16 * half + kThreads - 1) / kThreads;
    QkvPair qp[kItems];
    float2 rf[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int i = tid + k * kThreads, r = i / half, c = i % half;
      if (i < 16 * half && r < G) {
        const int hq = g * G + r;
        qkv_pair_load(p, b, hq * D + c, half, p.bias[0], hq * D + c, qp[k]);
        rf[k] = pos_ok ? cs[c] : make_float2(1.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int i = tid + k * kThreads, r = i / half, c = i % half;
      if (i >= 16 * half) break;
      float2 v = make_float2(0.f, 0.f);
      if (r < G) {
        v = qkv_pair_sum(p, qp[k]);
        if (pos_ok) {
          const float2 f = rf[k];
          v = make_float2(v.x * f.x - v.y * f.y, v.y * f.x + v.x * f.y);
        }
      }
      qtile[r * Sm::kQStride + c] = __float2half_rn(v.x);
      qtile[r * Sm::kQStride + half + c] = __float2half_rn(v.y);
    }
    const bool slot_here = n > 0 && L >= j0 && L < j1;
    if (n == 0 && tid == 0 && sp == 0 && g == 0) set_error(p.err, kDevPosition);
    if (slot_here) {
      __half* kd = p.kc + (size_t)b * p.Hkv * p.max_ctx * D + ((size_t)g * p.max_ctx + L) * D;
      __half* vd = p.vc + (size_t)b * p.Hkv * p.max_ctx * D + ((size_t)g * p.max_ctx + L) * D;
      const size_t nw = ((size_t)b * p.Hkv + g) * D;
      for (int i = tid; i < 2 * half; i += kThreads) {
        const bool is_k = i < half;
        const int c = is_k ? i : i - half;
        const int col = (is_k ? p.Hq + g : p.Hq + p.Hkv + g) * D + c;
        QkvPair kp;
        qkv_pair_load(p, b, col, half, is_k ? p.bias[1] : p.bias[2], g * D + c, kp);
        float2 v = qkv_pair_sum(p, kp);
        if (is_k && pos_ok) {
          const float2 f = cs[c];
          v = make_float2(v.x * f.x - v.y * f.y, v.y * f.x + v.x * f.y);
        }
        const __half h0 = __float2half_rn(v.x), h1 = __float2half_rn(v.y);
        __half* d = is_k ? kd : vd;
        d[c] = h0;
        d[half + c] = h1;
        __half* nwp = is_k ? p.k_new : p.v_new;
        if (nwp) {
          nwp[nw + c] = h0;
          nwp[nw + half + c] = h1;
        }
      }
      fence_proxy_async_global();   // before the tensor copy of slot L
    }
    __syncthreads();
  } else {
    // Q tile: rows 0..G-1 = query heads g*G.., rows G..15 zero
    for (int i = tid; i < 16 * kCPR; i += kThreads) {
      const int r = i / kCPR, ch = i % kCPR;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < G)
        v = *reinterpret_cast<const uint4*>(p.q16 + ((size_t)b * p.Hq + g * G + r) * D + ch * 8);
      *reinterpret_cast<uint4*>(qtile + r * Sm::kQStride + ch * 8) = v;
    }
  }
  if (tid == 0)
    for (; issued < kGroups - 1 && issued < ngroups; ++issued) load_group(issued);
  __syncthreads();   // the barriers are initialised before anyone waits on them

  const int grp = lane >> 2, tig = lane & 3;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float O[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
  const uint32_t qbase = smem_u32(qtile);
  const float sl2 = p.scale_log2;

  bool aborted = false;
  int gi = 0;
  for (; gi < ngroups; ++gi) {
    // group gi has landed (bounded wait); the block agrees on giving up, and
    // the barrier also frees group (gi-1) % kGroups for the next copy
    const bool ok = mbar_wait(&full[gi % kGroups], (uint32_t)(gi / kGroups) & 1u, p.err);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (tid == 0 && gi + kGroups - 1 < ngroups) load_group(gi + kGroups - 1);
    // this warp: tile gi*kTPG + warp/4 of the group, its slots 16*(warp%4)..
    const int jt = warp >> 2;
    const uint32_t kb = kv0 + ((gi % kGroups) * kTPG + jt) * 2 * Sm::kTile, vb = kb + Sm::kTile;
    const int64_t cs = j0 + (int64_t)(gi * kTPG + jt) * kTileSlots;
    const int nval = (int)max((int64_t)0, min((int64_t)kTileSlots, j1 - cs));
    const int r0 = (warp & 3) * 16;
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
      if (r0 + 16 > nval) {
        // slots past the split's end: their P is 0, but their V rows (other
        // slots' data) could hold non-finite values, so this warp zeroes its own
        for (int i = lane; i < 16 * kCPR; i += 32) {
          const int r = r0 + i / kCPR;
          if (r >= nval) st_shared_zero16(tile_addr(vb, r, i % kCPR));
        }
        fence_proxy_async_smem();   // before a later tensor copy into this tile
        __syncwarp();
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
  if (aborted) {
    // the copies already issued (groups gi .. gi + kGroups - 2) land before
    // the CTA exits; the status word already holds the timeout
    if (tid == 0)
      for (int g2 = gi; g2 < ngroups && g2 < gi + kGroups - 1; ++g2)
        mbar_wait(&full[g2 % kGroups], (uint32_t)(g2 / kGroups) & 1u, nullptr);
    return;
  }
  __syncthreads();      // every warp is done with the ring: the merge buffers reuse it

  // merge the warps' states in a fixed tree (1 -> 0, 3 -> 2, ..., then 2 -> 0, ...)
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
#pragma unroll
  for (int d = 1; d < kWarps; d *= 2) {   // warp w with w % 2d == d hands over to w - d
    float* bf = bufs + (warp / (2 * d)) * kBuf;
    if (warp % (2 * d) == d) put(bf);
    __syncthreads();
    if (warp % (2 * d) == 0) merge_from(bf);
    __syncthreads();
  }
  if (warp == 0) put(bufs);
  __syncthreads();

  // rows < G: attn (one split) or this split's fp32 partial
  for (int i = tid; i < G * D; i += kThreads) {
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

template <int D, int kGroups, int kTPG>
static cudaError_t launch_attn_batch_d(const DecodeAttnBatchParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nsplit, p.Hkv, p.B);
  cfg.blockDim = dim3(128 * kTPG);
  cfg.dynamicSmemBytes = BSmem<D, kGroups, kTPG>::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_attn_batch_kernel<D, kGroups, kTPG>, p);
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
    return p.deep ? launch_attn_batch_d<128, kGroupsDeep, kTpgDeep>(p, s)
                  : launch_attn_batch_d<128, kGroupsPair, kTpgPair>(p, s);
  if (p.D == 64)
    return p.deep ? launch_attn_batch_d<64, kGroupsDeep, kTpgDeep>(p, s)
                  : launch_attn_batch_d<64, kGroupsPair, kTpgPair>(p, s);
  return cudaErrorInvalidValue;
}

template <int D, int kGroups, int kTPG>
static cudaError_t configure_one() {
  return cudaFuncSetAttribute(decode_attn_batch_kernel<D, kGroups, kTPG>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)BSmem<D, kGroups, kTPG>::kBytes);
}

cudaError_t configure_decode_attn_batch() {
  cudaError_t e = configure_one<128, kGroupsDeep, kTpgDeep>();
  if (e == cudaSuccess) e = configure_one<128, kGroupsPair, kTpgPair>();
  if (e == cudaSuccess) e = configure_one<64, kGroupsDeep, kTpgDeep>();
  if (e == cudaSuccess) e = configure_one<64, kGroupsPair, kTpgPair>();
  return e;
}

}  // namespace blk
