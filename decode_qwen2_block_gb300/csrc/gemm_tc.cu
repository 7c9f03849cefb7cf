// Prefill projections on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// D[m, n] = sum_k A[m, k] * B[n, k]: A = activations [M, K] fp16, B = weights
// [N, K] fp16 (nn.Linear layout), both K-major; fp32 accumulation in TMEM.
//
// CTAs run as pairs (clusters of 2) on 256-row tiles with the 2-SM form of
// the MMA (tcgen05.mma.cta_group::2, M = 256): each CTA of the pair holds 128
// rows of A and half of the BN weight rows, the leader CTA issues the MMAs for
// both, and each SM's TMEM receives its own 128 rows of the result.  Per SM
// and K step this moves half of the weight tile through shared memory instead
// of all of it; with one-SM M = 128 MMAs the TMA writes plus the tensor core's
// reads of a 128 x 256 x 64 step (96 KB) already fill the 128 B/clock
// shared-memory port for longer than the MMA takes.
// One persistent CTA per SM, 10 warps:
//   warp 0   TMA producer (both CTAs): this CTA's 128x64 A tile and its
//            (BN/2)x64 part of the weight tile, 128-byte swizzle, into a ring
//            of shared-memory stages; the copies complete on the leader's
//            stage barrier, and a stage is refilled after the leader's MMAs
//            released it in both CTAs.  Weight tiles of the first stages are
//            issued before griddepcontrol.wait (they never depend on the
//            previous kernel).
//   warp 1   allocates TMEM (two accumulators of BN fp32 columns, in both SMs
//            of the pair); in the leader its lane 0 issues
//            tcgen05.mma.cta_group::2.kind::f16 (M=256, N=BN, K=16) four
//            times per stage; tcgen05.commit (multicast to the pair) frees the
//            stage and, after a tile's last stage, hands both accumulators to
//            the epilogues.
//   warps 2-9 epilogue (both CTAs): tcgen05.ld 32 columns at a time (thread =
//            tile row, two warps per TMEM lane quarter),
//            fused per projection:
//              QKV    + bias, RoPE on q/k pairs (i, i+D/2), q -> fp16 buffer,
//                     k/v -> cache slots cache_len + m and k_new / v_new
//              O      + residual (block input, fp16) -> h (fp32)
//              GATEUP B tile = 128 rows of W_gate over 128 rows of W_up,
//                     silu(gate) * up -> activation (fp16)
//              DOWN   + residual h (fp32) -> block output (fp16)
//            or, when the launcher splits K (every projection but GATEUP,
//            given a partial buffer), an fp32 partial per split that a
//            finishing kernel adds up in split order; then release the
//            accumulator, so the MMA of the next tile overlaps this epilogue.
// Few rows (batched decode): the A box covers M rounded up to 8 rows, an M
// tile that starts past M is not loaded, and epilogue warps whose rows all
// lie past M skip their math (those accumulator rows hold arbitrary values).
// Every mbarrier wait is bounded; on a timeout the CTA records an error,
// stops issuing work, waits (bounded) for what it already issued and frees
// its TMEM before returning.
#include <cuda.h>

#include "common.cuh"
#include "gemm_tc.h"

namespace blk {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int kEpiWarps = 8;   // two per TMEM lane quarter, splitting the columns
constexpr int kThreads = 64 + 32 * kEpiWarps;

// 2-D tile into this CTA's shared memory, completing on an mbarrier that may
// be in the other CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// Address of this CTA's shared variable `p` in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (SBO), start address in 16-byte units, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* p) {
  const uint64_t addr = (smem_u32(p) & 0x3FFFFu) >> 4;
  uint64_t d = addr;
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;            // version
  d |= (uint64_t)2 << 61;            // swizzle mode: 128B
  return d;
}

// Instruction descriptor, kind::f16: D f32, A/B f16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM, both SMs) [+]= A (256 rows: 128 in each CTA's shared memory at the
// offset of `a`) x B (N rows: N/2 in each CTA at the offset of `b`).
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives, once the MMAs issued so far complete, on the mbarrier at the offset
// of `bar` in both CTAs of the pair.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)), "h"((uint16_t)3)
      : "memory");
}

// Same, on this CTA's mbarrier only.
__device__ __forceinline__ void mma_commit_local(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
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
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void store_h32(__half* dst, const float* v) {
  // 32 fp16 values, dst 16-byte aligned
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
    d[j] = u;
  }
}

// Writes this warp's 32 rows x 32 columns (lane = row, v = its 32 values)
// as full-row pieces: the values go through `st` (this warp's staging area in
// shared memory, 32 * (row bytes + 16) bytes) and each store instruction then
// covers whole 64- or 128-byte row pieces instead of one 16-byte piece of 32
// different rows.  gdst: row 0's destination (16-byte aligned), ld: row
// pitch in bytes; rows >= nrows are not written.
template <bool F16>
__device__ __forceinline__ void store_rows_staged(uint8_t* st, const float* v, int lane,
                                                  uint8_t* gdst, size_t ld, int nrows) {
  constexpr int kRowB = F16 ? 64 : 128;
  constexpr int kStride = kRowB + 16;
  uint4* s4 = reinterpret_cast<uint4*>(st + lane * kStride);
  if constexpr (F16) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 u;
      __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[8 * k + 2 * i], v[8 * k + 2 * i + 1]);
      s4[k] = u;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      s4[k] = make_uint4(__float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]),
                         __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
  }
  __syncwarp();
  constexpr int kLpr = kRowB / 16;   // lanes per row piece
  constexpr int kRpi = 32 / kLpr;    // rows per store instruction
  const int rr = lane / kLpr, cc = lane % kLpr;
#pragma unroll
  for (int i = 0; i < 32 / kRpi; ++i) {
    const int row = i * kRpi + rr;
    const uint4 val = *reinterpret_cast<const uint4*>(st + row * kStride + cc * 16);
    if (row < nrows) *reinterpret_cast<uint4*>(gdst + row * ld + cc * 16) = val;
  }
  __syncwarp();   // the staging area is reused by the warp's next call
}

template <int BN>
struct Cfg {
  static constexpr int kBHalf = BN / 2;                  // weight rows per CTA of the pair
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = kBHalf * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (192 * 1024) / kStageBytes;
  static constexpr int kTmemCols = 2 * BN;  // two accumulators
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024 + 256;
};

// A work unit is (N tile nt, M tile pair mp, K split ks): the CTA of rank r
// in the pair takes M tile 2 mp + r.
template <int EPI, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcGemmParams p) {
  using C = Cfg<BN>;
  constexpr int kBBox = 64;                      // rows per weight tensor-map box
  constexpr int kBBoxes = C::kBHalf / kBBox;     // boxes per CTA and stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;   // [2]
  uint64_t* tempty = tfull + 2;           // [2], counted in the leader
  uint64_t* drain = tempty + 2;           // [1], used only on the abort path
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (p.K + BK - 1) / BK;

  const uint32_t rank = cluster_rank();          // 0: the leader, which issues the MMAs
  const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;   // pair index and count
  const int mpairs = (p.tiles_m + 1) / 2;
  // K is split S ways when the launcher chose to (every epilogue but gate/up):
  // each split writes an fp32 partial that a later kernel adds up
  const int S = EPI == kTcGateUp ? 1 : p.splits;
  const int KBs = (KB + S - 1) / S;   // K blocks per split
  const int units = mpairs * p.tiles_n * S;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);   // the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {   // the same columns in both SMs of the pair
    asm volatile(
        "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(tmem_slot)),
        "r"((uint32_t)C::kTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the leader's barriers exist before the peer's copies complete on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tmA);
      prefetch_tmap(&p.tmB[0]);
      if (EPI == kTcQKV || EPI == kTcGateUp) prefetch_tmap(&p.tmB[1]);
      if (EPI == kTcQKV) prefetch_tmap(&p.tmB[2]);
      int it = 0;
      bool waited = false;
      const uint32_t a_bytes = (uint32_t)(p.a_rows > 0 ? p.a_rows : BM) * BK * 2;
      for (int u = cl; u < units && !*abort_flag; u += ncl) {
        const int t = u / S, ks = u % S;
        const int mt = (t % mpairs) * 2 + (int)rank, nt = t / mpairs;
        const int m0 = mt * BM, n0 = nt * (EPI == kTcGateUp ? BN / 2 : BN);
        const int kb1 = min(KB, (ks + 1) * KBs);
        // A tiles that start past M are not loaded: their accumulator rows
        // are never stored.  Both CTAs' copies complete on the leader's barrier.
        const bool a_mine = m0 < p.M;
        const uint32_t tx = 2 * C::kBBytes +
                            ((t % mpairs) * 2 * BM < p.M ? a_bytes : 0) +
                            (((t % mpairs) * 2 + 1) * BM < p.M ? a_bytes : 0);
        for (int kb = ks * KBs; kb < kb1; ++kb, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&empty[s], ((it / C::kStages) & 1) ^ 1, p.err)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* sa = smem + (size_t)s * C::kStageBytes;
          uint8_t* sb = sa + C::kABytes;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], tx);
          const uint32_t fb = cluster_addr(&full[s], 0);
          // this CTA's weight rows: GATEUP leader W_gate, peer W_up (same rows);
          // otherwise rows n0 + rank * BN/2 ...
#pragma unroll
          for (int bx = 0; bx < kBBoxes; ++bx) {
            const CUtensorMap* mb;
            int row;
            if (EPI == kTcGateUp) {
              mb = &p.tmB[rank];
              row = n0 + bx * kBBox;
            } else {
              int seg = 0;
              row = n0 + (int)rank * C::kBHalf + bx * kBBox;
              if (EPI == kTcQKV) {
                while (seg < 2 && row >= p.seg_rows[seg]) row -= p.seg_rows[seg++];
              }
              mb = &p.tmB[seg];
            }
            tma_load_2d_pair(sb + bx * (kBBox * BK * 2), mb, kb * BK, row, fb);
          }
          if (!waited) {  // activations come from the previous kernel
            griddep_wait();
            griddep_launch();
            waited = true;
          }
          if (a_mine) tma_load_2d_pair(sa, &p.tmA, kb * BK, m0, fb);
        }
      }
      if (!waited) {
        griddep_wait();
        griddep_launch();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_f16(2 * BM, BN);
      int it = 0, tcount = 0;
      bool issued = false;
      for (int u = cl; u < units && !*abort_flag; u += ncl, ++tcount) {
        const int acc = tcount & 1;
        if (!mbar_wait(&tempty[acc], ((tcount >> 1) & 1) ^ 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int ks = u % S, kb0 = ks * KBs, kb1 = min(KB, kb0 + KBs);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err)) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint8_t* sa = smem + (size_t)s * C::kStageBytes;
          const uint64_t da = smem_desc_sw128(sa);
          const uint64_t db = smem_desc_sw128(sa + C::kABytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // +32 bytes per K step inside the swizzle atom
            mma_f16_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, (kb != kb0) || (k != 0));
          issued = true;
          mma_commit_pair(&empty[s]);
        }
        if (*abort_flag) break;
        mma_commit_pair(&tfull[acc]);
      }
      if (*abort_flag && issued) {  // let issued MMAs finish before TMEM is freed
        mma_commit_local(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    griddep_wait();
    griddep_launch();
    // Thread = tile row.  Warps 2..9 read TMEM lane quarter warp % 4; the two
    // warps of a quarter take alternate 32-column chunks.  Each warp issues
    // the global loads its chunks need (residual, RoPE factors) before it
    // reads the accumulator, so their latency overlaps.
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int e = (warp - 2) >> 2;       // which half of the chunks
    const int row_in_tile = q * 32 + lane;
    int tcount = 0;
    for (int u = cl; u < units; u += ncl, ++tcount) {
      const int acc = tcount & 1;
      const int t = u / S, ks = u % S;
      const int mt = (t % mpairs) * 2 + (int)rank, nt = t / mpairs;
      const int m = mt * BM + row_in_tile;
      const bool row_ok = m < p.M;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      float v0[32], v1[32];
      // On the CTA's last tile every stage has been consumed once the
      // accumulator is full, so the stages serve as store staging areas.
      const bool staged = u + ncl >= units;
      uint8_t* stg = smem + (warp - 2) * (32 * 144);
      const int row0 = mt * BM + q * 32;              // this warp's first row
      const int nrows = min(32, p.M - row0);

      if (S > 1) {
        // split K: this split's fp32 partial [ks][M][N]; the finishing kernel
        // (split-K reduction, QKV finish, or RMSNorm of the summed rows) adds
        // the partials in split order and applies the epilogue
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], (tcount >> 1) & 1, p.err))) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int n0 = nt * BN;
        float* part = p.part + (size_t)ks * p.M * p.N;
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          const int c0 = 32 * e + 64 * c;
          if (row0 >= p.M) break;   // warp-uniform: no row of this warp exists
          tmem_ld32(tbase + c0, v0);
          if (n0 + c0 >= p.N) continue;
          if (staged) {
            store_rows_staged<false>(
                stg, v0, lane, reinterpret_cast<uint8_t*>(part + (size_t)row0 * p.N + n0 + c0),
                (size_t)p.N * 4, nrows);
            continue;
          }
          if (!row_ok) continue;
          float4* dst = reinterpret_cast<float4*>(part + (size_t)m * p.N + n0 + c0);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
        }
      } else if constexpr (EPI == kTcQKV) {
        const int D = p.D, half = D / 2;
        const int n0 = nt * BN;
        const int64_t pos = row_ok ? p.pos[m] : 0;
        // (head, chunk) items of this tile, alternating between the two warps
        const int chunks = half / 32, items = (BN / D) * chunks;
        bool waited = false;
        for (int it2 = e; it2 < items; it2 += 2) {
          const int hh = it2 / chunks, c0 = (it2 % chunks) * 32;
          const int hd = n0 / D + hh;  // head index over q | k | v
          const __half* bias;
          int local;
          if (hd < p.Hq) { bias = p.bias[0]; local = hd; }
          else if (hd < p.Hq + p.Hkv) { bias = p.bias[1]; local = hd - p.Hq; }
          else { bias = p.bias[2]; local = hd - p.Hq - p.Hkv; }
          const bool rope = hd < p.Hq + p.Hkv;
          // bias of columns c0 + lane and half + c0 + lane (shared by all rows;
          // broadcast with shuffles), loaded before the accumulator
          const float b0 = bias ? __half2float(bias[local * D + c0 + lane]) : 0.f;
          const float b1 = bias ? __half2float(bias[local * D + half + c0 + lane]) : 0.f;
          // this row's 32 rotation factors, loaded before the accumulator
          float4 cs4[16];
          if (rope && row_ok && pos >= 0 && pos < p.rope_len) {
            const float4* src = reinterpret_cast<const float4*>(p.rope + (size_t)pos * half + c0);
#pragma unroll
            for (int k = 0; k < 16; ++k) cs4[k] = __ldg(src + k);
          } else {
            if (rope && row_ok) set_error(p.err, kDevPosition);
#pragma unroll
            for (int k = 0; k < 16; ++k) cs4[k] = make_float4(1.f, 0.f, 1.f, 0.f);
          }
          if (!waited) {
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], (tcount >> 1) & 1, p.err))) {
              *abort_flag = 1;
              break;
            }
            tc_fence_after();
            waited = true;
          }
          tmem_ld32(tbase + hh * D + c0, v0);
          tmem_ld32(tbase + hh * D + half + c0, v1);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v0[i] += __shfl_sync(0xffffffffu, b0, i);
            v1[i] += __shfl_sync(0xffffffffu, b1, i);
          }
          if (!row_ok && !staged) continue;
          if (rope) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float4 c = cs4[i >> 1];
              const float cx = (i & 1) ? c.z : c.x, sy = (i & 1) ? c.w : c.y;
              const float a = v0[i], b = v1[i];
              v0[i] = a * cx - b * sy;
              v1[i] = b * cx + a * sy;
            }
          }
          // batched decode: row m is sequence m, its K/V go to its own cache
          const bool kv_rows = hd >= p.Hq && p.cache_lens != nullptr;
          if (staged && !kv_rows) {
            uint8_t* g;
            size_t ld;
            __half* nw = nullptr;
            if (hd < p.Hq) {
              g = reinterpret_cast<uint8_t*>(p.q16 + ((size_t)row0 * p.Hq + hd) * D);
              ld = (size_t)p.Hq * D * 2;
            } else {
              const bool is_k = hd < p.Hq + p.Hkv;
              nw = is_k ? p.k_new : p.v_new;
              g = reinterpret_cast<uint8_t*>((is_k ? p.kc : p.vc) +
                                             ((size_t)local * p.max_ctx + p.cache_len + row0) * D);
              ld = (size_t)D * 2;
            }
            store_rows_staged<true>(stg, v0, lane, g + c0 * 2, ld, nrows);
            store_rows_staged<true>(stg, v1, lane, g + (half + c0) * 2, ld, nrows);
            if (nw) {
              uint8_t* g2 = reinterpret_cast<uint8_t*>(nw + ((size_t)row0 * p.Hkv + local) * D);
              const size_t ld2 = (size_t)p.Hkv * D * 2;
              store_rows_staged<true>(stg, v0, lane, g2 + c0 * 2, ld2, nrows);
              store_rows_staged<true>(stg, v1, lane, g2 + (half + c0) * 2, ld2, nrows);
            }
          } else if (!row_ok) {
            // rows past M hold nothing to store
          } else if (hd < p.Hq) {
            __half* dst = p.q16 + ((size_t)m * p.Hq + hd) * D;
            store_h32(dst + c0, v0);
            store_h32(dst + half + c0, v1);
          } else {
            const bool is_k = hd < p.Hq + p.Hkv;
            __half* cache = is_k ? p.kc : p.vc;
            __half* nw = is_k ? p.k_new : p.v_new;
            int64_t slot = p.cache_len + m;
            if (p.cache_lens) {
              slot = p.cache_lens[m];
              cache += (size_t)m * p.seq_stride;
            }
            if (slot >= 0 && slot < p.max_ctx) {
              __half* dst = cache + ((size_t)local * p.max_ctx + slot) * D;
              store_h32(dst + c0, v0);
              store_h32(dst + half + c0, v1);
            } else if (c0 == 0) {
              set_error(p.err, kDevPosition);
            }
            if (nw) {
              __half* d2 = nw + ((size_t)m * p.Hkv + local) * D;
              store_h32(d2 + c0, v0);
              store_h32(d2 + half + c0, v1);
            }
          }
        }
        if (!waited) {   // no item for this warp: still wait so the release is ordered
          if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], (tcount >> 1) & 1, p.err))) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
        }
      } else if constexpr (EPI == kTcGateUp) {
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], (tcount >> 1) & 1, p.err))) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int j0 = nt * (BN / 2);
        // a warp whose 32 rows all lie past M has nothing to store (its
        // accumulator rows come from unloaded, arbitrary A rows)
        for (int c0 = 32 * e; c0 < BN / 2 && row0 < p.M; c0 += 64) {
          tmem_ld32(tbase + c0, v0);
          tmem_ld32(tbase + BN / 2 + c0, v1);
#pragma unroll
          for (int i = 0; i < 32; ++i) v0[i] = silu(v0[i]) * v1[i];
          if (staged && j0 + c0 + 32 <= p.N) {
            store_rows_staged<true>(
                stg, v0, lane, reinterpret_cast<uint8_t*>(p.out16 + (size_t)row0 * p.ldo + j0 + c0),
                (size_t)p.ldo * 2, nrows);
            continue;
          }
          if (!row_ok) continue;
          __half* dst = p.out16 + (size_t)m * p.ldo + j0 + c0;
          if (j0 + c0 + 32 <= p.N) {
            store_h32(dst, v0);
          } else {   // ragged last columns (unrolled: v0 stays in registers)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (j0 + c0 + i < p.N) dst[i] = __float2half_rn(v0[i]);
          }
        }
      } else {
        const int n0 = nt * BN;
        constexpr int kCh = BN / 64;   // chunks per warp: c0 = 32 e + 64 c
        // loads row m's residual for chunk c0 (zeros outside the output)
        auto load_res = [&](int c0, float* rv) {
          const bool ok = row_ok && n0 + c0 < p.N;
          const size_t o = (size_t)m * p.ldo + n0 + c0;
          if constexpr (EPI == kTcResidF32) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float f[8];
              h8_to_f32(ok ? __ldg(reinterpret_cast<const uint4*>(p.res16 + o) + j)
                           : make_uint4(0u, 0u, 0u, 0u), f);
#pragma unroll
              for (int t2 = 0; t2 < 8; ++t2) rv[8 * j + t2] = f[t2];
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 f = ok ? __ldg(reinterpret_cast<const float4*>(p.res32 + o) + j)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
              rv[4 * j] = f.x; rv[4 * j + 1] = f.y; rv[4 * j + 2] = f.z; rv[4 * j + 3] = f.w;
            }
          }
        };
        auto store_out = [&](int c0, const float* v) {
          const size_t o = (size_t)m * p.ldo + n0 + c0;
          if constexpr (EPI == kTcResidF32) {
            float4* dst = reinterpret_cast<float4*>(p.out32 + o);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            store_h32(p.out16 + o, v);
          }
        };
        {
          // two chunks at a time: their residuals are loaded before the
          // accumulator is read
          bool waited = false;
#pragma unroll
          for (int c2 = 0; c2 < kCh; c2 += 2) {
            float rv[2][32];
#pragma unroll
            for (int c = 0; c < 2; ++c)
              if (c2 + c < kCh) load_res(32 * e + 64 * (c2 + c), rv[c]);
            if (!waited) {
              if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], (tcount >> 1) & 1, p.err))) {
                *abort_flag = 1;
                break;
              }
              tc_fence_after();
              waited = true;
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              if (c2 + c >= kCh) break;
              const int c0 = 32 * e + 64 * (c2 + c);
              tmem_ld32(tbase + c0, v0);
              if (n0 + c0 >= p.N) continue;
#pragma unroll
              for (int i = 0; i < 32; ++i) v0[i] += rv[c][i];
              if (staged) {
                if constexpr (EPI == kTcResidF32)
                  store_rows_staged<false>(
                      stg, v0, lane,
                      reinterpret_cast<uint8_t*>(p.out32 + (size_t)row0 * p.ldo + n0 + c0),
                      (size_t)p.ldo * 4, nrows);
                else
                  store_rows_staged<true>(
                      stg, v0, lane,
                      reinterpret_cast<uint8_t*>(p.out16 + (size_t)row0 * p.ldo + n0 + c0),
                      (size_t)p.ldo * 2, nrows);
              } else if (row_ok) {
                store_out(c0, v0);
              }
            }
          }
          if (!waited) break;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(&tempty[acc], 0));   // leader's count
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA of the pair leaves while the other may still use its shared
  // memory, its barriers or its TMEM
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"((uint32_t)C::kTmemCols)
                 : "memory");
  }
}

// out16[m, n] = fp16(sum_j part[j][m, n] + res32[m, n]), splits added in
// order; four columns per element, two elements (a grid stride apart) per
// thread with every load of both issued before any add.  MAXS (>= S) sizes
// the register arrays: 4 for the usual 2-4 splits keeps a thread near 40
// registers, so that a whole grid is resident at once.
template <int MAXS>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part,
                                                            int S, int64_t MN,
                                                            const float* __restrict__ res32,
                                                            __half* __restrict__ out16) {
  griddep_wait();
  griddep_launch();
  const int64_t n4 = MN / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n4; i0 += 2 * stride) {
    float4 r[2], q[2][MAXS];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int64_t i = i0 + e * stride;
      if (i >= n4) break;
      r[e] = __ldg(reinterpret_cast<const float4*>(res32) + i);
#pragma unroll
      for (int j = 0; j < MAXS; ++j)
        if (j < S) q[e][j] = __ldcg(reinterpret_cast<const float4*>(part + (size_t)j * MN) + i);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int64_t i = i0 + e * stride;
      if (i >= n4) break;
      float4 a = q[e][0];   // splits added in ascending order, then the residual
#pragma unroll
      for (int j = 1; j < MAXS; ++j)
        if (j < S) { a.x += q[e][j].x; a.y += q[e][j].y; a.z += q[e][j].z; a.w += q[e][j].w; }
      uint2 o;
      *reinterpret_cast<__half2*>(&o.x) = __floats2half2_rn(a.x + r[e].x, a.y + r[e].y);
      *reinterpret_cast<__half2*>(&o.y) = __floats2half2_rn(a.z + r[e].z, a.w + r[e].w);
      reinterpret_cast<uint2*>(out16)[i] = o;
    }
  }
}

// Finishes a K-split QKV projection: element (row m, head hd, pair i) of the
// fused q | k | v output is the sum of the split partials (split order) plus
// the bias, rotated by RoPE for q and k heads, then stored exactly as the
// GEMM's own QKV epilogue does (q16; K/V into the cache slot and k_new/v_new).
template <int MAXS>
__global__ void __launch_bounds__(64) qkv_finish_kernel(const __grid_constant__ TcGemmParams p) {
  griddep_wait();
  griddep_launch();
  const int hd = blockIdx.x, m = blockIdx.y;
  const int D = p.D, half = D / 2;
  const size_t MN = (size_t)p.M * p.N;
  int local;
  const __half* bias;
  if (hd < p.Hq) { bias = p.bias[0]; local = hd; }
  else if (hd < p.Hq + p.Hkv) { bias = p.bias[1]; local = hd - p.Hq; }
  else { bias = p.bias[2]; local = hd - p.Hq - p.Hkv; }
  const bool rope = hd < p.Hq + p.Hkv;
  const int64_t pos = p.pos[m];
  const bool pos_ok = pos >= 0 && pos < p.rope_len;
  if (rope && !pos_ok && threadIdx.x == 0) set_error(p.err, kDevPosition);
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const size_t c0 = (size_t)m * p.N + (size_t)hd * D + i, c1 = c0 + half;
    // every split's pair is loaded before any is added (one round trip)
    float qa[MAXS], qb[MAXS];
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
      if (s < p.splits) {
        qa[s] = __ldcg(p.part + s * MN + c0);
        qb[s] = __ldcg(p.part + s * MN + c1);
      }
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
      if (s < p.splits) {
        a += qa[s];
        b += qb[s];
      }
    if (bias) {
      a += __half2float(bias[local * D + i]);
      b += __half2float(bias[local * D + half + i]);
    }
    if (rope && pos_ok) {
      const float2 cs = p.rope[(size_t)pos * half + i];
      const float a2 = a * cs.x - b * cs.y, b2 = b * cs.x + a * cs.y;
      a = a2;
      b = b2;
    }
    const __half ha = __float2half_rn(a), hb = __float2half_rn(b);
    if (hd < p.Hq) {
      __half* dst = p.q16 + ((size_t)m * p.Hq + hd) * D;
      dst[i] = ha;
      dst[half + i] = hb;
      continue;
    }
    const bool is_k = hd < p.Hq + p.Hkv;
    __half* cache = is_k ? p.kc : p.vc;
    __half* nw = is_k ? p.k_new : p.v_new;
    int64_t slot = p.cache_len + m;
    if (p.cache_lens) {
      slot = p.cache_lens[m];
      cache += (size_t)m * p.seq_stride;
    }
    if (slot >= 0 && slot < p.max_ctx) {
      __half* dst = cache + ((size_t)local * p.max_ctx + slot) * D;
      dst[i] = ha;
      dst[half + i] = hb;
    } else if (i == 0) {
      set_error(p.err, kDevPosition);
    }
    if (nw) {
      __half* d2 = nw + ((size_t)m * p.Hkv + local) * D;
      d2[i] = ha;
      d2[half + i] = hb;
    }
  }
}

}  // namespace

// ---------------------------------------------------------------- host side

cudaError_t launch_splitk_reduce(const TcGemmParams& p, int num_sms, cudaStream_t s) {
  if (p.splits < 1 || p.splits > 16) return cudaErrorInvalidValue;
  const int64_t MN = (int64_t)p.M * p.N;
  const int64_t n4 = MN / 4;
  const int maxs = p.splits <= 4 ? 4 : (p.splits <= 8 ? 8 : 16);
  // two elements per thread; no more blocks than are resident at once
  static int resident[3] = {0, 0, 0};
  int& res = resident[maxs == 4 ? 0 : (maxs == 8 ? 1 : 2)];
  if (res == 0) {
    int nb = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &nb,
        maxs == 4 ? splitk_reduce_kernel<4> : (maxs == 8 ? splitk_reduce_kernel<8>
                                                         : splitk_reduce_kernel<16>),
        256, 0);
    res = (e == cudaSuccess && nb > 0 ? nb : 1) * num_sms;
  }
  int grid = (int)((n4 + 511) / 512);
  if (grid > res) grid = res;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid < 1 ? 1 : grid);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float* part = p.part;
  if (maxs == 4)
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<4>, part, p.splits, MN, p.res32, p.out16);
  if (maxs == 8)
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<8>, part, p.splits, MN, p.res32, p.out16);
  return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<16>, part, p.splits, MN, p.res32, p.out16);
}

cudaError_t launch_qkv_finish(const TcGemmParams& p, cudaStream_t s) {
  if (p.splits < 2 || p.splits > 16 || !p.part || p.D / 2 > 64) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq + 2 * p.Hkv, p.M);
  cfg.blockDim = dim3(p.D / 2);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.splits <= 4) return cudaLaunchKernelEx(&cfg, qkv_finish_kernel<4>, p);
  if (p.splits <= 8) return cudaLaunchKernelEx(&cfg, qkv_finish_kernel<8>, p);
  return cudaLaunchKernelEx(&cfg, qkv_finish_kernel<16>, p);
}

// cuTensorMapEncodeTiled, resolved through the runtime so that the library
// does not link libcuda (it must load on machines without a driver).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

int make_tmap_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                 int box_rows) {
  const EncodeTiledFn encode = encode_tiled();
  if (!encode) return -1;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(
      map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_tmap_3d(CUtensorMap* map, const void* base, const int64_t* dims,
                 const int64_t* strides, const int* box) {
  const EncodeTiledFn encode = encode_tiled();
  if (!encode) return -1;
  cuuint64_t d[3] = {(cuuint64_t)dims[0], (cuuint64_t)dims[1], (cuuint64_t)dims[2]};
  cuuint64_t st[2] = {(cuuint64_t)strides[0], (cuuint64_t)strides[1]};
  cuuint32_t bx[3] = {(cuuint32_t)box[0], (cuuint32_t)box[1], (cuuint32_t)box[2]};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), d, st,
                            bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_tmap_4d(CUtensorMap* map, const void* base, const int64_t* dims,
                 const int64_t* strides, const int* box) {
  const EncodeTiledFn encode = encode_tiled();
  if (!encode) return -1;
  cuuint64_t d[4] = {(cuuint64_t)dims[0], (cuuint64_t)dims[1], (cuuint64_t)dims[2],
                     (cuuint64_t)dims[3]};
  cuuint64_t st[3] = {(cuuint64_t)strides[0], (cuuint64_t)strides[1], (cuuint64_t)strides[2]};
  cuuint32_t bx[4] = {(cuuint32_t)box[0], (cuuint32_t)box[1], (cuuint32_t)box[2],
                      (cuuint32_t)box[3]};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), d, st,
                            bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_tmap_rows8(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int cbs,
                    int* is3d) {
  const EncodeTiledFn encode = encode_tiled();
  if (!encode) return -1;
  CUresult r;
  if (K % 64 == 0) {
    // (64 columns, rows, K / 64 column blocks): one copy moves 8 rows x cbs blocks
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(K / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
    cuuint32_t box[3] = {64, 8, (cuuint32_t)cbs};
    cuuint32_t estr[3] = {1, 1, 1};
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *is3d = 1;
  } else {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, 8};
    cuuint32_t estr[2] = {1, 1};
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *is3d = 0;
  }
  return r == CUDA_SUCCESS ? 0 : -1;
}

int make_tmap_codes(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                    int cbs, int* is3d) {
  const EncodeTiledFn encode = encode_tiled();
  if (!encode) return -1;
  CUresult r;
  if (row_bytes % 128 == 0) {
    // (128 bytes, rows, row_bytes / 128 blocks): one copy moves 8 rows x cbs blocks
    cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)(row_bytes / 128)};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, 128};
    cuuint32_t box[3] = {128, 8, (cuuint32_t)cbs};
    cuuint32_t estr[3] = {1, 1, 1};
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *is3d = 1;
  } else {
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128, 8};
    cuuint32_t estr[2] = {1, 1};
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *is3d = 0;
  }
  return r == CUDA_SUCCESS ? 0 : -1;
}

template <int EPI, int BN>
static cudaError_t launch_tc(TcGemmParams& p, int num_sms, cudaStream_t s, bool pdl) {
  using C = Cfg<BN>;
  p.tiles_m = (p.M + BM - 1) / BM;
  const int bn_out = EPI == kTcGateUp ? BN / 2 : BN;
  p.tiles_n = (p.N + bn_out - 1) / bn_out;
  p.num_tiles = p.tiles_m * p.tiles_n;
  const int mpairs = (p.tiles_m + 1) / 2;
  int units = mpairs * p.tiles_n;
  // co-resident pairs: one CTA per SM
  static int max_pairs = 0;
  if (max_pairs == 0) {
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(2 * 64);
    q.blockDim = dim3(kThreads);
    q.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute qa[1];
    qa[0].id = cudaLaunchAttributeClusterDimension;
    qa[0].val.clusterDim.x = 2;
    qa[0].val.clusterDim.y = 1;
    qa[0].val.clusterDim.z = 1;
    q.attrs = qa;
    q.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<EPI, BN>, &q) != cudaSuccess || n < 1)
      n = num_sms / 2;
    max_pairs = n < num_sms / 2 ? n : num_sms / 2;
  }
  p.splits = 1;
  if (EPI != kTcGateUp && p.part && p.max_splits > 1) {
    // split K so that the units fill the co-resident pairs (8+ K blocks each)
    int S = max_pairs / units;
    S = S < 1 ? 1 : (S > p.max_splits ? p.max_splits : S);
    const int KB = (p.K + BK - 1) / BK;
    while (S > 1 && KB / S < 8) --S;
    p.splits = S;
    units *= S;
  }
  const int pairs = units < max_pairs ? units : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = 2;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<EPI, BN>, p);
}

cudaError_t launch_tc_gemm(TcGemmParams& p, int epi, int num_sms, cudaStream_t s,
                           bool pdl) {
  switch (epi) {
    case kTcQKV: return launch_tc<kTcQKV, 128>(p, num_sms, s, pdl);
    case kTcResidF32: return launch_tc<kTcResidF32, 128>(p, num_sms, s, pdl);
    case kTcGateUp: return launch_tc<kTcGateUp, 256>(p, num_sms, s, pdl);
    default: return launch_tc<kTcResidOutF16, 256>(p, num_sms, s, pdl);
  }
}

template <int EPI, int BN>
static cudaError_t configure_one() {
  return cudaFuncSetAttribute(tc_gemm_kernel<EPI, BN>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<BN>::kSmem);
}

cudaError_t configure_tc_gemm_kernels() {
  cudaError_t e;
  if ((e = configure_one<kTcQKV, 128>())) return e;
  if ((e = configure_one<kTcResidF32, 128>())) return e;
  if ((e = configure_one<kTcGateUp, 256>())) return e;
  return configure_one<kTcResidOutF16, 256>();
}

}  // namespace blk
