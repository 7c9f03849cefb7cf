// Causal GQA attention for prefill / prefill_kv on the tensor cores.
//
// CTA = (query head h, block of 64 new rows): 4 consumer warps own 16 query
// rows each; a producer warp streams 64-slot K and V tiles of kv head
// h / (Hq/Hkv) from the cache (128-byte-swizzled tensor copies, two stages,
// mbarrier full/empty pairs).  Per tile, each warp computes S = Q K^T with
// mma.sync m16n8k16 (fp16 in, fp32 accumulate; Q fragments stay in
// registers), applies the causal mask (new row t sees slots [0, L + t]),
// updates an online softmax in base 2 (log2(e)/sqrt(D) folded into q) and
// accumulates O += P V (P rounded to fp16, V fragments via ldmatrix.trans).
// Tiles a warp cannot see are skipped; cache rows past the last valid slot
// are zeroed in shared memory before use so stale values never reach P V.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {
namespace {

constexpr int kWarps = 4;            // consumer warps, 16 query rows each
constexpr int kRows = 16 * kWarps;   // query rows per CTA
constexpr int kSlots = 64;           // cache slots per K/V tile
constexpr int kStages = 2;

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

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

// 16-byte chunk `ch` of row `r` of a 64-row tile stored as 128-byte-swizzled
// half tiles of 64 columns (8 KB each).
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int ch) {
  const int half = ch >> 3, c = ch & 7;
  return base + half * 8192 + r * 128 + ((c ^ (r & 7)) << 4);
}

template <int D>
struct Smem {
  static constexpr int kTile = kSlots * D * 2;        // K or V tile bytes
  static constexpr int kStage = 2 * kTile;            // K + V
  static constexpr int kQStride = D + 8;              // halves, padded rows
  static constexpr int kQBytes = kRows * kQStride * 2;
  static constexpr size_t kBytes = (size_t)kStages * kStage + kQBytes + 64 + 1024;
  static_assert(kStages * 16 + 4 <= 64, "barrier area");
};

template <int D>
__global__ void __launch_bounds__((kWarps + 1) * 32)
    prefill_attn_mma_kernel(const __grid_constant__ PrefillAttnParams p) {
  using S = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  __half* qs = reinterpret_cast<__half*>(smem + kStages * S::kStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * S::kStage + S::kQBytes);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int nqb = (p.T + kRows - 1) / kRows;
  const int qb = nqb - 1 - (int)blockIdx.y;  // longest rows first
  const int t0 = qb * kRows;
  const int G = p.Hq / p.Hkv, g = h / G;
  const int64_t L = p.cache_len;
  const int64_t n_keys = L + min(p.T, t0 + kRows);  // slots the CTA can see
  const int ntiles = (int)((n_keys + kSlots - 1) / kSlots);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      griddep_wait();    // the new K/V rows come from the previous kernel
      griddep_launch();
      int issued = 0;
      for (int j = 0; j < ntiles; ++j, ++issued) {
        const int s = j % kStages;
        if (*abort_flag) break;
        if (j >= kStages && !mbar_wait(&empty[s], ((j / kStages) - 1) & 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], S::kStage);
        uint8_t* st = ring + (size_t)s * S::kStage;
        const int y = (int)(g * p.max_ctx + (int64_t)j * kSlots);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          tma_load_2d(st + hh * 8192, &p.tm_k, hh * 64, y, &full[s]);
          tma_load_2d(st + S::kTile + hh * 8192, &p.tm_v, hh * 64, y, &full[s]);
        }
      }
      for (int k = max(0, issued - kStages); k < issued; ++k)
        mbar_wait(&full[k % kStages], (k / kStages) & 1, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();
  griddep_launch();
  const int grp = lane >> 2, tig = lane & 3;
  const int r_lo = t0 + warp * 16;          // first query row of this warp
  // Q tile of this warp -> shared (padded rows) -> A fragments.
  {
    __half* qw = qs + warp * 16 * S::kQStride;
    constexpr int cpr = D / 8;  // 16-byte chunks per row
    for (int i = lane; i < 16 * cpr; i += 32) {
      const int r = i / cpr, c = i % cpr;
      const int t = r_lo + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < p.T)
        v = *reinterpret_cast<const uint4*>(p.q16 + ((size_t)t * p.Hq + h) * D + c * 8);
      // scale by log2(e)/sqrt(D) (folded into q once, in fp32, rounded back)
      __half2* hv = reinterpret_cast<__half2*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(hv[e]);
        hv[e] = __floats2half2_rn(f.x * p.scale_log2, f.y * p.scale_log2);
      }
      *reinterpret_cast<uint4*>(qw + r * S::kQStride + c * 8) = v;
    }
    __syncwarp();
  }
  uint32_t qf[D / 16][4];
  {
    const uint32_t qbase = smem_u32(qs + warp * 16 * S::kQStride);
    const int m = lane >> 3, rr = (m & 1) * 8 + (lane & 7);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      ldsm_x4(qbase + (rr * S::kQStride + ks * 16 + (m >> 1) * 8) * 2, qf[ks]);
  }

  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float O[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
  const int64_t last_row_slot = L + min(p.T - 1, r_lo + 15);  // furthest slot this warp sees
  const int64_t valid_end = L + p.T;                          // slots >= this are never valid

  for (int j = 0; j < ntiles; ++j) {
    const int s = j % kStages;
    // After a timed-out wait the loop runs on without touching the tile (so
    // every warp still reaches the barrier below) and stores nothing.
    bool ok = !*abort_flag;
    if (ok && !mbar_wait(&full[s], (j / kStages) & 1, p.err)) {
      *abort_flag = 1;
      ok = false;
    }
    uint8_t* st = ring + (size_t)s * S::kStage;
    const uint32_t kb = smem_u32(st), vb = kb + S::kTile;
    const int64_t js = (int64_t)j * kSlots;
    // Zero cache rows past the last valid slot (only in the last tile); each
    // warp clears 16 rows, then all consumers sync before using the tile.
    if (js + kSlots > valid_end) {
      const int first_bad = (int)(valid_end - js);
      for (int i = lane; i < 16 * (D / 8) && ok; i += 32) {
        const int r = warp * 16 + i / (D / 8), ch = i % (D / 8);
        if (r >= first_bad) {
          *reinterpret_cast<uint4*>(st + (tile_addr(kb, r, ch) - kb)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(st + (tile_addr(vb, r, ch) - kb)) = make_uint4(0, 0, 0, 0);
        }
      }
      named_sync(1, kWarps * 32);
    }
    if (ok && r_lo < p.T && js <= last_row_slot) {
      // S = Q K^T over 64 slots: 8 n-tiles of 8 slots
      float Sc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) Sc[nt][0] = Sc[nt][1] = Sc[nt][2] = Sc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {   // pairs of n-tiles
          uint32_t bk[4];
          const int m = lane >> 3;
          const int r = np * 16 + (m >> 1) * 8 + (lane & 7);
          ldsm_x4(tile_addr(kb, r, ks * 2 + (m & 1)), bk);
          mma16816(Sc[2 * np], qf[ks], bk[0], bk[1]);
          mma16816(Sc[2 * np + 1], qf[ks], bk[2], bk[3]);
        }
      }
      // causal mask + online softmax (rows grp and grp + 8)
      const bool need_mask = js + kSlots - 1 > L + r_lo || r_lo + 16 > p.T;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (need_mask) {
            const int64_t slot = js + nt * 8 + 2 * tig + (e & 1);
            const int64_t t = r_lo + grp + 8 * (e >> 1);
            if (slot > L + t || t >= p.T) Sc[nt][e] = -INFINITY;
          }
          mx[e >> 1] = fmaxf(mx[e >> 1], Sc[nt][e]);
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
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        O[dn][0] *= corr[0]; O[dn][1] *= corr[0];
        O[dn][2] *= corr[1]; O[dn][3] *= corr[1];
      }
      uint32_t pa[8][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mn = m_r[e >> 1];
          pv[e] = (Sc[nt][e] == -INFINITY || mn == -INFINITY) ? 0.f : exp2f(Sc[nt][e] - mn);
          l_r[e >> 1] += pv[e];
        }
        pa[nt][0] = pack_h2(pv[0], pv[1]);
        pa[nt][1] = pack_h2(pv[2], pv[3]);
      }
      // O += P V: 4 k-steps of 16 slots
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t afr[4] = {pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1]};
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t bv[4];
          const int m = lane >> 3;
          const int r = kk * 16 + (m & 1) * 8 + (lane & 7);
          ldsm_x4_t(tile_addr(vb, r, dp * 2 + (m >> 1)), bv);
          mma16816(O[2 * dp], afr, bv[0], bv[1]);
          mma16816(O[2 * dp + 1], afr, bv[2], bv[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  if (*abort_flag) return;
  // normalise and store rows grp and grp + 8 of this warp
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    l_r[h2] += __shfl_xor_sync(0xffffffffu, l_r[h2], 1);
    l_r[h2] += __shfl_xor_sync(0xffffffffu, l_r[h2], 2);
  }
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int t = r_lo + grp + 8 * h2;
    if (t >= p.T) continue;
    const float inv = 1.f / l_r[h2];
    __half* dst = p.attn16 + (size_t)t * p.Hq * D + h * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn)
      *reinterpret_cast<__half2*>(dst + dn * 8 + 2 * tig) =
          __floats2half2_rn(O[dn][2 * h2] * inv, O[dn][2 * h2 + 1] * inv);
  }
}

template <int D>
cudaError_t launch_mma(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq, (p.T + kRows - 1) / kRows);
  cfg.blockDim = dim3((kWarps + 1) * 32);
  cfg.dynamicSmemBytes = Smem<D>::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prefill_attn_mma_kernel<D>, p);
}

}  // namespace

cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  if (p.D == 128) return launch_mma<128>(p, s, pdl);
  if (p.D == 64) return launch_mma<64>(p, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t configure_prefill_attn() {
  cudaError_t e = cudaFuncSetAttribute(prefill_attn_mma_kernel<128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Smem<128>::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_attn_mma_kernel<64>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem<64>::kBytes);
}

}  // namespace blk
