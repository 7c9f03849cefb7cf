// Causal GQA attention for prefill / prefill_kv on the 5th-generation tensor
// cores (the FAttention step of the TopOp decoder block: softmax(q k^T /
// sqrt(D)) v over slots [0, L + t] for new row t).
//
// CTA = (query head h, block of 128 new rows), 6 warps:
//   warp 0   TMA producer: the Q block once (3-D view of q [T, Hq, D]), then
//            128-slot K and V tiles of kv head h / (Hq/Hkv) into two stages.
//            The K/V tensor maps end at slot L + T, so slots past the last
//            valid one arrive as zeros (stale cache contents never reach PV).
//   warp 1   allocates TMEM (S: 128 columns, O: D columns) and its lane 0
//            issues the MMAs (tcgen05.mma.cta_group::1.kind::f16, M = 128):
//            S_j = Q K_j^T (N = 128, K = D), then O += P_j V_j (N = D,
//            K = 128; V is the MN-major B operand).  S_{j+1} is issued as
//            soon as the softmax has read S_j, so it overlaps that softmax.
//   warps 2-5 softmax (thread = query row): read S_j from TMEM, scale by
//            log2(e)/sqrt(D), causal mask, online softmax in base 2 (rescale
//            O in TMEM when the row maximum grows), write P_j (fp16) to shared
//            memory in the MMA's K-major layout; at the end O / l -> attn (fp16).
// Every wait is bounded; on a timeout the CTA records an error, stops, lets
// issued MMAs finish and frees its TMEM before returning.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace blk {
namespace {

constexpr int kRows = 128;        // query rows per CTA (MMA M)
constexpr int kSlots = 128;       // cache slots per K/V tile (MMA N of S, K of PV)
constexpr int kStages = 2;
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

template <int D>
struct Smem {
  static constexpr int kQBytes = kRows * D * 2;            // [D/64][128 rows][128 B]
  static constexpr int kKVTile = kSlots * D * 2;            // K or V: [D/64][128 slots][128 B]
  static constexpr int kStage = 2 * kKVTile;
  static constexpr int kPBytes = kRows * kSlots * 2;        // [2][128 rows][128 B]
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQBytes;
  static constexpr int kPOff = kKVOff + kStages * kStage;
  static constexpr int kBarOff = kPOff + kPBytes;
  static constexpr size_t kBytes = (size_t)kBarOff + 256 + 1024;
  static constexpr uint32_t kTmemCols = 256;                 // S (128) + O (D), power of two
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_tc_kernel(const __grid_constant__ PrefillAttnParams p) {
  using Sm = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Sm::kQOff;
  uint8_t* sKV = smem + Sm::kKVOff;
  uint8_t* sP = smem + Sm::kPOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;           // [2]
  uint64_t* kv_empty = bars + 3;          // [2]
  uint64_t* s_full = bars + 5;            // S_j in TMEM
  uint64_t* s_free = bars + 6;            // the softmax has read S_j
  uint64_t* p_full = bars + 7;            // P_j in shared memory, O rescaled
  uint64_t* o_done = bars + 8;            // O += P_j V_j complete
  uint64_t* drain = bars + 9;             // abort path
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int nqb = (p.T + kRows - 1) / kRows;
  const int qb = nqb - 1 - (int)blockIdx.y;  // longest rows first
  const int t0 = qb * kRows;
  const int G = p.Hq / p.Hkv, g = h / G;
  const int64_t L = p.cache_len;
  const int64_t n_keys = L + min(p.T, t0 + kRows);  // slots this block can see
  const int ntiles = (int)((n_keys + kSlots - 1) / kSlots);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
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
  const uint32_t tS = tmem, tO = tmem + kSlots;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      griddep_wait();    // q and the new K/V rows come from the previous kernel
      griddep_launch();
      mbar_arrive_expect_tx(q_full, Sm::kQBytes);
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh)
        tma_load_3d(sQ + hh * (kRows * 128), &p.tm_q, hh * 64, h, t0, q_full);
      int issued = 0;
      for (int j = 0; j < ntiles; ++j, ++issued) {
        const int s = j % kStages;
        if (*abort_flag) break;
        if (j >= kStages && !mbar_wait(&kv_empty[s], ((j / kStages) - 1) & 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[s], Sm::kStage);
        uint8_t* st = sKV + (size_t)s * Sm::kStage;
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          tma_load_3d(st + hh * (kSlots * 128), &p.tm_k, hh * 64, j * kSlots, g, &kv_full[s]);
          tma_load_3d(st + Sm::kKVTile + hh * (kSlots * 128), &p.tm_v, hh * 64, j * kSlots, g,
                      &kv_full[s]);
        }
      }
      // copies still in flight land before shared memory goes away
      mbar_wait(q_full, 0, nullptr);
      for (int k = max(0, issued - kStages); k < issued; ++k)
        mbar_wait(&kv_full[k % kStages], (k / kStages) & 1, nullptr);
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
        if (!mbar_wait(&kv_full[s], (j / kStages) & 1, p.err)) return false;
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
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < ntiles && ok; ++j) {
        if (j + 1 < ntiles && !issue_s(j + 1)) { ok = false; break; }
        if (!mbar_wait(p_full, j & 1, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = smem_u32(sKV + (size_t)(j % kStages) * Sm::kStage + Sm::kKVTile);
        const uint32_t pb = smem_u32(sP);
#pragma unroll
        for (int kk = 0; kk < kSlots / 16; ++kk) {   // O += P_j V_j over 16 slots at a time
          const uint64_t a = desc_kmajor(pb + (kk >> 2) * (kRows * 128)) + ((kk & 3) * 32 >> 4);
          const uint64_t b = desc_mnmajor(vb + kk * 16 * 128);
          mma(tO, a, b, id_o, (j | kk) != 0);
        }
        commit(o_done);
        commit(&kv_empty[j % kStages]);
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
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // The tcgen05.ld/st below are warp-collective (.sync.aligned): every
    // decision before one of them is made uniform across the warp.
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.err));
    };
    for (int j = 0; j < ntiles; ++j) {
      if (!wait_all(s_full, j & 1)) { ok = false; break; }
      tc_fence_after();
      float sv[kSlots];
#pragma unroll
      for (int c = 0; c < kSlots; c += 32) tmem_ld32(tS + lane_off + c, sv + c);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);   // S may be overwritten by S_{j+1}
      const int64_t js = (int64_t)j * kSlots;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kSlots; ++c) {
        float v = sv[c] * p.scale_log2;
        if (!row_ok || js + c > last) v = -INFINITY;
        sv[c] = v;
        mx = fmaxf(mx, v);
      }
      // The reference maximum of a row moves (and O, l are rescaled) only
      // when the row maximum grew by more than 2^8 since it last moved: P stays
      // <= 256 and the final 1 / l normalisation makes the choice exact.  The
      // decision is per warp (the rescale below is warp-collective); moving a
      // row's reference up to its current maximum is always valid.
      const bool need = (m == -INFINITY) ? (mx != -INFINITY) : (mx - m > kRescaleLog2);
      const bool move = __any_sync(0xffffffffu, need);
      const float mn = move ? fmaxf(m, mx) : m;
      const float alpha = (m == -INFINITY || mn == m) ? 1.f : exp2f(m - mn);
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < kSlots; ++c) {
        const float e = (sv[c] == -INFINITY) ? 0.f : exp2f(sv[c] - mn);
        sv[c] = e;
        sum += e;
      }
      l = l * alpha + sum;
      m = mn;
      if (j > 0) {
        // PV_{j-1} must be complete before O is rescaled and P overwritten
        if (!wait_all(o_done, (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (move) {
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
      }
      // P_j (fp16) into the K-major 128-byte-swizzled layout: [slot half][row][128 B]
#pragma unroll
      for (int c = 0; c < kSlots / 8; ++c) {
        uint4 u;
        __half2* hp = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) hp[e] = __floats2half2_rn(sv[8 * c + 2 * e], sv[8 * c + 2 * e + 1]);
        const int half = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4*>(sP + half * (kRows * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = u;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // for the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && wait_all(o_done, (ntiles - 1) & 1)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __half* dst = p.attn16 + ((size_t)t * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        float ov[32];
        tmem_ld32(tO + lane_off + c, ov);
        tmem_wait_ld();
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            __half2* hp = reinterpret_cast<__half2*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              hp[e] = __floats2half2_rn(ov[8 * k + 2 * e] * inv, ov[8 * k + 2 * e + 1] * inv);
            d4[k] = u;
          }
        }
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

template <int D>
cudaError_t launch_tc(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq, (p.T + kRows - 1) / kRows);
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

cudaError_t launch_prefill_attn(const PrefillAttnParams& p, cudaStream_t s, bool pdl) {
  if (p.D == 128) return launch_tc<128>(p, s, pdl);
  if (p.D == 64) return launch_tc<64>(p, s, pdl);
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
