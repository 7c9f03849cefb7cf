// Causal GQA attention for prefill / prefill_kv on the 5th-generation tensor
// cores (the FAttention step of the TopOp decoder block: softmax(q k^T /
// sqrt(D)) v over slots [0, L + t] for new row t).
//
// CTA = (query head h, block of 128 new rows, chunk of that block's 128-slot
// tiles), 6 warps:
//   warp 0   TMA producer: the Q block once (3-D view of q [T, Hq, D]), then
//            the chunk's K and V tiles of kv head h / (Hq/Hkv) into three
//            stages; a K stage frees when S_j is computed, a V stage when
//            PV_j is.  The K/V tensor maps end at slot L + T, so slots past the
//            last valid one arrive as zeros (stale cache contents never reach PV).
//   warp 1   allocates TMEM (S: 128 columns, O: D columns, two P buffers of 64)
//            and its lane 0 issues the MMAs (tcgen05.mma.cta_group::1.kind::f16,
//            M = 128): S_j = Q K_j^T (N = 128, K = D, both from shared
//            memory), then O += P_j V_j (N = D, K = 128; P is the A operand
//            read from TMEM, V the MN-major B operand).  S_{j+1} is issued as
//            soon as the softmax has read S_j, so it overlaps that softmax.
//   warps 2-5 softmax (thread = query row): read S_j from TMEM, causal mask on
//            tiles that cross the diagonal, online softmax in base 2 with lazy
//            rescaling of O in TMEM, P_j (fp16 pairs) into TMEM buffer j % 2;
//            at the end O / l -> attn.
// A block whose tiles are split over several CTAs (chunks, so that the long
// blocks of the causal triangle do not set the kernel's duration) publishes
// per-chunk partials (O, m, l in fp32) that attn_merge_kernel, launched next,
// combines.
// Every wait is bounded; on a timeout the CTA records an error, stops, lets
// issued MMAs finish and frees its TMEM before returning.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {
namespace {

constexpr int kRows = 128;        // query rows per CTA (MMA M)
constexpr int kSlots = 128;       // cache slots per K/V tile (MMA N of S, K of PV)
constexpr int kStages = 3;       // K/V stages
constexpr int kThreads = 192;
constexpr float kRescaleLog2 = 8.f;   // see the softmax: lazy rescaling threshold

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major, 128-byte swizzle: 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  uint64_t d = (saddr & 0x3FFFFu) >> 4;
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// MN-major, 128-byte swizzle: 64 MN elements per 128-byte row, 8 rows (K) per
// atom; the next 64 MN elements 16 KB further (LBO), the next 8 K rows 1 KB
// further (SBO).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) {
  uint64_t d = (saddr & 0x3FFFFu) >> 4;
  d |= (uint64_t)(16384 >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// kind::f16 instruction descriptor: D f32, A/B f16, A K-major, B K-major or
// MN-major, M x N.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int b_mn) {
  return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

// Same with the A operand (M x 16, K-major: row i = TMEM lane i, element
// pairs packed in 32-bit columns) read from TMEM at a_tmem.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, "
      "%9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, "
      "%24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]),
        "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, "
      "%9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, "
      "%25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {   // 2^x; ex2(-inf) = +0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct Smem {
  static constexpr int kQBytes = kRows * D * 2;            // [D/64][128 rows][128 B]
  static constexpr int kKVTile = kSlots * D * 2;            // K or V: [D/64][128 slots][128 B]
  static constexpr int kStage = 2 * kKVTile;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQBytes;
  static constexpr int kBarOff = kKVOff + kStages * kStage;
  static constexpr size_t kBytes = (size_t)kBarOff + 256 + 1024;
  // TMEM columns: S (128 fp32), O (D fp32), two P buffers (128 fp16 packed in
  // 64 columns each); allocated as a power of two.
  static constexpr uint32_t kSCol = 0, kOCol = kSlots, kPCol = kSlots + 128;
  static constexpr uint32_t kTmemCols = 512;
};

// Partial result of one chunk of a query block (fp32): per 32-row quarter q
// its O (not normalised) as [D/4][32 rows] float4 at q * D * 32 floats (one
// contiguous block of D * 128 bytes), then at 128 * D floats, per quarter, the
// rows' reference maxima m (log2 units) and sums l: [4][m 32 | l 32].
template <int D>
__device__ __forceinline__ float* part_ptr(const PrefillAttnParams& p, int h, int qb, int ch) {
  return p.part + ((size_t)(h * p.nqb + qb) * p.max_chunks + ch) * (size_t)(kRows * (D + 2));
}

__device__ __forceinline__ void store_row32(__half* d, const float* v, float inv) {
  uint4* d4 = reinterpret_cast<uint4*>(d);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 u;
    __half2* hp = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      hp[e] = __floats2half2_rn(v[8 * k + 2 * e] * inv, v[8 * k + 2 * e + 1] * inv);
    d4[k] = u;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_tc_kernel(const __grid_constant__ PrefillAttnParams p) {
  using Sm = Smem<D>;
  const int h = blockIdx.x;
  const int qb = p.nqb - 1 - (int)blockIdx.y;  // longest rows first
  const int ch = blockIdx.z;                     // chunk of the block's tiles
  const int t0 = qb * kRows;
  const int64_t L = p.cache_len;
  const int64_t n_keys = L + min(p.T, t0 + kRows);  // slots this block can see
  const int ntot = (int)((n_keys + kSlots - 1) / kSlots);
  // with a sliding window the block's first row sees slots from window_lo on
  const int jlo = (int)(window_lo(p.window, L + t0) / kSlots);
  const int nch = (ntot - jlo + p.chunk_tiles - 1) / p.chunk_tiles;
  if (ch >= nch) return;                         // (uniform over the CTA)
  const int j0 = jlo + ch * p.chunk_tiles;       // first tile of this CTA
  const int nt = min(ntot, j0 + p.chunk_tiles) - j0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Sm::kQOff;
  uint8_t* sKV = smem + Sm::kKVOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;                  // [kStages] K_j in stage j % kStages
  uint64_t* k_empty = k_full + kStages;         // [kStages] S_j complete: K stage free
  uint64_t* v_full = k_empty + kStages;         // [kStages]
  uint64_t* v_empty = v_full + kStages;         // [kStages] PV_j complete: V stage free
  uint64_t* s_full = v_empty + kStages;         // S_j in TMEM
  uint64_t* s_free = s_full + 1;                // the softmax has read S_j
  uint64_t* p_full = s_free + 1;                // [2] P_j in TMEM buffer j % 2 (O rescaled)
  uint64_t* o_done = p_full + 2;                // [2] O += P_j V_j complete (j % 2)
  uint64_t* drain = o_done + 2;                 // abort path
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv, g = h / G;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p_full[b], 4);
      mbar_init(&o_done[b], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(tmem_slot)),
        "r"(Sm::kTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem + Sm::kSCol, tO = tmem + Sm::kOCol, tP = tmem + Sm::kPCol;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      griddep_wait();    // q and the new K/V rows come from the previous kernel
      griddep_launch();
      mbar_arrive_expect_tx(q_full, Sm::kQBytes);
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh)
        tma_load_3d(sQ + hh * (kRows * 128), &p.tm_q, hh * 64, h, t0, q_full);
      // K_j's stage frees when S_j is complete, V_j's when PV_j is: K runs
      // up to two tiles ahead of the softmax.
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j % kStages;
        const uint32_t par = ((j / kStages) - 1) & 1;
        uint8_t* st = sKV + (size_t)s * Sm::kStage;
        const int y = (j0 + j) * kSlots;
        if (*abort_flag) break;
        if (j >= kStages && !mbar_wait(&k_empty[s], par, p.err)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], Sm::kKVTile);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh)
          tma_load_3d(st + hh * (kSlots * 128), &p.tm_k, hh * 64, y, g, &k_full[s]);
        ++issued_k;
        if (j >= kStages && !mbar_wait(&v_empty[s], par, p.err)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&v_full[s], Sm::kKVTile);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh)
          tma_load_3d(st + Sm::kKVTile + hh * (kSlots * 128), &p.tm_v, hh * 64, y, g,
                      &v_full[s]);
        ++issued_v;
      }
      // copies still in flight land before shared memory goes away
      mbar_wait(q_full, 0, nullptr);
      for (int k = max(0, issued_k - kStages); k < issued_k; ++k)
        mbar_wait(&k_full[k % kStages], (k / kStages) & 1, nullptr);
      for (int k = max(0, issued_v - kStages); k < issued_v; ++k)
        mbar_wait(&v_full[k % kStages], (k / kStages) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc(kRows, kSlots, 0);
      constexpr uint32_t id_o = idesc(kRows, D, 1);
      bool ok = mbar_wait(q_full, 0, p.err);
      bool issued = false;
      auto issue_s = [&](int j) -> bool {   // S_j = Q K_j^T
        const int s = j % kStages;
        if (!mbar_wait(&k_full[s], (j / kStages) & 1, p.err)) return false;
        if (j > 0 && !mbar_wait(s_free, (j - 1) & 1, p.err)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(sKV + (size_t)s * Sm::kStage);
        const uint32_t qb_ = smem_u32(sQ);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * (kRows * 128);
          const uint64_t a = desc_kmajor(qb_ + off) + ((ks & 3) * 32 >> 4);
          const uint64_t b = desc_kmajor(kb + off) + ((ks & 3) * 32 >> 4);
          mma(tS, a, b, id_s, ks != 0);
        }
        issued = true;
        commit(s_full);
        commit(&k_empty[s]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nt && ok; ++j) {
        if (j + 1 < nt && !issue_s(j + 1)) { ok = false; break; }
        const int b = j & 1;
        if (!mbar_wait(&p_full[b], (j >> 1) & 1, p.err)) { ok = false; break; }
        if (!mbar_wait(&v_full[j % kStages], (j / kStages) & 1, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = smem_u32(sKV + (size_t)(j % kStages) * Sm::kStage + Sm::kKVTile);
#pragma unroll
        for (int kk = 0; kk < kSlots / 16; ++kk) {   // O += P_j V_j over 16 slots at a time
          const uint64_t bd = desc_mnmajor(vb + kk * 16 * 128);
          mma_ts(tO, tP + b * (kSlots / 2) + kk * 8, bd, id_o, (j | kk) != 0);
        }
        commit(&o_done[b]);
        commit(&v_empty[j % kStages]);
      }
      if (!ok) {
        *abort_flag = 1;
        if (issued) {   // let issued MMAs finish before TMEM is freed
          commit(drain);
          mbar_wait(drain, 0, nullptr);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q * 32 + lane;            // query row in the block
    const int t = t0 + r;
    const bool row_ok = t < p.T;
    const int64_t last = L + t;             // last slot row t may see
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // The tcgen05.ld/st below are warp-collective (.sync.aligned): every
    // decision before one of them is made uniform across the warp.
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.err));
    };
    // With a sliding window the block's first tile can hold slots below
    // every row's window: their P is 0, but 0 * NaN is NaN in the PV MMA, so
    // a non-finite value left in such a slot is zeroed in shared memory
    // before PV_0 is issued (it waits for this warp's arrive on p_full[0]).
    if (p.window > 0 && ch == 0) {
      const int64_t lo0 = window_lo(p.window, L + t0), js0 = (int64_t)j0 * kSlots;
      if (lo0 > js0) {
        if (!wait_all(&v_full[0], 0)) ok = false;
        if (ok && js0 + r < lo0) {
          uint8_t* vrow = sKV + Sm::kKVTile + (size_t)r * 128;
#pragma unroll
          for (int hh = 0; hh < D / 64; ++hh)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vrow + hh * (kSlots * 128) + c * 16) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
    }
    for (int j = 0; j < nt && ok; ++j) {
      if (!wait_all(s_full, j & 1)) { ok = false; break; }
      tc_fence_after();
      float sv[kSlots];
#pragma unroll
      for (int c = 0; c < kSlots; c += 32) tmem_ld32(tS + lane_off + c, sv + c);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);   // S may be overwritten by S_{j+1}
      const int64_t js = (int64_t)(j0 + j) * kSlots;
      if (js + kSlots - 1 > L + t0) {         // the tile crosses the causal diagonal
        const int64_t d = last - js;
        const int lim = d < -1 ? -1 : (d > kSlots - 1 ? kSlots - 1 : (int)d);
#pragma unroll
        for (int c = 0; c < kSlots; ++c)
          if (c > lim) sv[c] = -INFINITY;
      }
      if (p.window > 0) {                     // slots before the row's window
        const int64_t d = window_lo(p.window, last) - js;
        const int lim = d < 0 ? 0 : (d > kSlots ? kSlots : (int)d);
#pragma unroll
        for (int c = 0; c < kSlots; ++c)
          if (c < lim) sv[c] = -INFINITY;
      }
      float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < kSlots; c += 4) {
        a0 = fmaxf(a0, sv[c]);
        a1 = fmaxf(a1, sv[c + 1]);
        a2 = fmaxf(a2, sv[c + 2]);
        a3 = fmaxf(a3, sv[c + 3]);
      }
      const float mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * sl2;   // log2 units
      // The reference maximum of a row moves (and O, l are rescaled) only
      // when the row maximum grew by more than 2^8 since it last moved: P stays
      // <= 256 and the final 1 / l normalisation makes the choice exact.  The
      // decision is per warp (the rescale below is warp-collective); moving a
      // row's reference up to its current maximum is always valid.
      const bool need = (m == -INFINITY) ? (mx != -INFINITY) : (mx - m > kRescaleLog2);
      const bool move = __any_sync(0xffffffffu, need);
      const float mn = move ? fmaxf(m, mx) : m;
      const float alpha = (m == -INFINITY || mn == m) ? 1.f : ex2(m - mn);
      const float nref = (mn == -INFINITY) ? 0.f : -mn;
      // P buffer j % 2 is free once PV_{j-2} is complete
      if (j >= 2 && !wait_all(&o_done[j & 1], ((j - 2) >> 1) & 1)) { ok = false; break; }
      // P_j (fp16, slot pairs packed in 32-bit columns: row r = TMEM lane r, the
      // MMA's A operand layout) into TMEM buffer j % 2
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      uint32_t pk[kSlots / 2];
#pragma unroll
      for (int c = 0; c < kSlots / 8; ++c) {
        float e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = ex2(fmaf(sv[8 * c + k], sl2, nref));
        s0 += e[0] + e[4];
        s1 += e[1] + e[5];
        s2 += e[2] + e[6];
        s3 += e[3] + e[7];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __half2 h2 = __floats2half2_rn(e[2 * k], e[2 * k + 1]);
          pk[4 * c + k] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      const uint32_t tPj = tP + (j & 1) * (kSlots / 2) + lane_off;
      tmem_st32(tPj, reinterpret_cast<const float*>(pk));
      tmem_st32(tPj + 32, reinterpret_cast<const float*>(pk + 32));
      l = l * alpha + ((s0 + s1) + (s2 + s3));
      m = mn;
      if (move && j > 0) {
        // PV_{j-1} must be complete before O is rescaled
        if (!wait_all(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          float ov[32];
          tmem_ld32(tO + lane_off + c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= alpha;
          tmem_st32(tO + lane_off + c, ov);
        }
        tmem_wait_st();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[j & 1]);
    }
    if (ok && wait_all(&o_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1)) {
      tc_fence_after();
      __half* dst = p.attn16 + ((size_t)t * p.Hq + h) * D;
      if (nch == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          float ov[32];
          tmem_ld32(tO + lane_off + c, ov);
          tmem_wait_ld();
          if (row_ok) store_row32(dst + c, ov, inv);
        }
      } else {
        // Several chunks: publish this chunk's partial for attn_merge_kernel.
        float* P = part_ptr<D>(p, h, qb, ch);
        float4* Oq = reinterpret_cast<float4*>(P + q * D * 32);
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          float ov[32];
          tmem_ld32(tO + lane_off + c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            Oq[(c / 4 + k) * 32 + lane] =
                make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
        }
        P[kRows * D + q * 64 + lane] = m;
        P[kRows * D + q * 64 + 32 + lane] = l;
      }
    } else {
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(Sm::kTmemCols)
                 : "memory");
  }
}

// Merges the partials of every block whose tiles were split over several
// CTAs: O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c, M = max_c m_c, as
// an online merge in chunk order with explicit roundings (the same bits on
// every run).  CTA = (block (h, qb), 32 output columns), thread = row: the
// D/32 column groups of a block are separate CTAs so that the merge spreads
// over four times as many SMs.
template <int D>
__global__ void __launch_bounds__(kRows)
    attn_merge_kernel(const __grid_constant__ PrefillAttnParams p) {
  const int h = blockIdx.x, qb = blockIdx.y;
  const int t0 = qb * kRows;
  const int64_t n_keys = p.cache_len + min(p.T, t0 + kRows);
  const int ntot = (int)((n_keys + kSlots - 1) / kSlots);
  const int jlo = (int)(window_lo(p.window, p.cache_len + t0) / kSlots);
  const int nch = (ntot - jlo + p.chunk_tiles - 1) / p.chunk_tiles;
  if (nch <= 1) return;                      // written by the attention kernel
  griddep_wait();
  griddep_launch();
  const int r = threadIdx.x, grp = blockIdx.z;
  const int q = r >> 5, lane = r & 31;
  float M = -INFINITY, lt = 0.f, acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  auto add = [&](const float4* v, float mc, float lc) {
    if (mc == -INFINITY) return;             // no slot of this chunk is visible
    const float mn = fmaxf(M, mc);
    const float so = (M == -INFINITY) ? 0.f : ex2(M - mn);
    const float w = ex2(mc - mn);
    lt = __fmaf_rn(w, lc, __fmul_rn(lt, so));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[4 * k] = __fmaf_rn(w, v[k].x, __fmul_rn(acc[4 * k], so));
      acc[4 * k + 1] = __fmaf_rn(w, v[k].y, __fmul_rn(acc[4 * k + 1], so));
      acc[4 * k + 2] = __fmaf_rn(w, v[k].z, __fmul_rn(acc[4 * k + 2], so));
      acc[4 * k + 3] = __fmaf_rn(w, v[k].w, __fmul_rn(acc[4 * k + 3], so));
    }
    M = mn;
  };
  auto load = [&](int c2, float4* v, float& mc, float& lc) {
    const float* P = part_ptr<D>(p, h, qb, c2);
    const float4* o4 = reinterpret_cast<const float4*>(P + q * D * 32);
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ldcg(o4 + (grp * 8 + k) * 32 + lane);
    mc = __ldcg(P + kRows * D + q * 64 + lane);
    lc = __ldcg(P + kRows * D + q * 64 + 32 + lane);
  };
  for (int c2 = 0; c2 < nch; c2 += 2) {      // two chunks' loads in flight
    float4 va[8], vb[8];
    float ma, la, mb = -INFINITY, lb = 0.f;
    load(c2, va, ma, la);
    if (c2 + 1 < nch) load(c2 + 1, vb, mb, lb);
    add(va, ma, la);
    if (c2 + 1 < nch) add(vb, mb, lb);
  }
  const int t = t0 + r;
  if (t < p.T) {
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    store_row32(p.attn16 + ((size_t)t * p.Hq + h) * D + grp * 32, acc, inv);
  }
}

template <int D>
cudaError_t launch_tc(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq, p.nqb, p.grid_chunks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<D>::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prefill_attn_tc_kernel<D>, p);
}

}  // namespace

int prefill_attn_max_chunks(int64_t T, int Hq, int num_sms) {
  const int64_t nqb = (T + kRows - 1) / kRows;
  const int64_t need = (2 * (int64_t)num_sms + Hq * nqb - 1) / (Hq * nqb);
  return (int)(need > 4 ? need : 4);
}

size_t prefill_attn_part_bytes(int64_t T, int Hq, int D, int num_sms) {
  const int64_t nqb = (T + kRows - 1) / kRows;
  return (size_t)(Hq * nqb) * prefill_attn_max_chunks(T, Hq, num_sms) * kRows * (D + 2) * 4;
}

// Chooses the chunk length C (tiles per CTA): the estimated time is the
// number of CTA waves times C, plus four tiles for publishing the partials
// and the merge kernel when blocks are split (measured: at T = 1024 splitting
// the 8-tile blocks in two gains nothing); ties go to the longer chunk.
void plan_prefill_attn(PrefillAttnParams& p, int num_sms) {
  const int64_t L = p.cache_len;
  p.nqb = (p.T + kRows - 1) / kRows;
  auto tiles = [&](int qb) {
    return (int)((L + min(p.T, (qb + 1) * kRows) + kSlots - 1) / kSlots) -
           (int)(window_lo(p.window, L + qb * kRows) / kSlots);
  };
  int nmax = 0;   // the most tiles any block sees (the last block without a window)
  for (int qb = 0; qb < p.nqb; ++qb) nmax = max(nmax, tiles(qb));
  double best = 1e300;
  int best_c = nmax, prev = -1;
  for (int k = 1; k <= p.max_chunks; ++k) {
    const int C = (nmax + k - 1) / k;
    if (C == prev) continue;
    prev = C;
    int64_t items = 0;
    for (int qb = 0; qb < p.nqb; ++qb) items += (tiles(qb) + C - 1) / C;
    items *= p.Hq;
    const int64_t waves = (items + num_sms - 1) / num_sms;
    const double cost = (double)waves * C + (C < nmax ? 4.0 : 0.0);
    if (cost < best) {
      best = cost;
      best_c = C;
    }
  }
  p.chunk_tiles = best_c;
  p.grid_chunks = (nmax + best_c - 1) / best_c;
}

cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  if (p.grid_chunks < 1 || p.grid_chunks > p.max_chunks || p.chunk_tiles < 1)
    return cudaErrorInvalidValue;
  if (p.grid_chunks > 1 && !p.part) return cudaErrorInvalidValue;
  if (p.D == 128) return launch_tc<128>(p, s, pdl);
  if (p.D == 64) return launch_tc<64>(p, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_merge(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  if (p.grid_chunks <= 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq, p.nqb, p.D / 32);
  cfg.blockDim = dim3(kRows);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.D == 128) return cudaLaunchKernelEx(&cfg, attn_merge_kernel<128>, p);
  if (p.D == 64) return cudaLaunchKernelEx(&cfg, attn_merge_kernel<64>, p);
  return cudaErrorInvalidValue;
}

cudaError_t configure_prefill_attn() {
  cudaError_t e = cudaFuncSetAttribute(prefill_attn_tc_kernel<128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Smem<128>::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_attn_tc_kernel<64>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)Smem<64>::kBytes);
}

}  // namespace blk
