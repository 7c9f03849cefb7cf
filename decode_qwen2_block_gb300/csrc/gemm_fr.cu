// Few-row projections of batched decode on the 5th-generation tensor cores.
//
// Y[m, n] = sum_k X[m, k] W[n, k] for a handful of activation rows (one per
// sequence of a decode batch, M <= 128) against an nn.Linear weight W [N, K].
// The operands are swapped against the prefill GEMM (gemm_tc.cu): W's rows
// are the MMA's M side (128 per CTA, every one an output column) and X's rows
// its N side (M padded to 32, 64 or 128), so no MMA row is padding and the
// bytes a CTA streams are its share of the weights plus X's columns of its K
// range.  Y^T = W X^T sits in TMEM with one lane per weight row and one
// column per activation row.
//
// One CTA per (128-row weight tile, K split), 6 warps; the launcher splits K
// only as far as the units still fit one wave (every projection of the 1.5B
// shape runs in one; gate/up of a 11008-wide MLP has 172 tiles, two waves):
//   warp 0   TMA producer: per 64-column K block, the tile's two 64-row
//            weight boxes and X's box (npad rows; rows past M arrive as
//            zeros) into a ring of 6 stages, 128-byte swizzle.  The weight
//            boxes of the first stages are issued before griddepcontrol.wait
//            (they never depend on the previous kernel).
//   warp 1   allocates npad TMEM columns; its lane 0 issues
//            tcgen05.mma.cta_group::1.kind::f16 (M = 128, N = npad, K = 16,
//            both operands K-major in shared memory) four times per stage,
//            commits the stage back to the producer and, after the last, the
//            accumulator to the epilogue.
//   warps 2-5 epilogue, thread = weight row (TMEM lane quarter warp % 4):
//            PART    this split's fp32 partial [split][M][N]: for each
//                    activation row a warp stores 32 consecutive columns
//                    (128 bytes).  A finishing kernel adds the splits in
//                    split order: the batched attention for QKV, the split-K
//                    RMSNorm for o_proj, the split-K reduction for down.
//            GATEUP  the tile is 64 rows of W_gate (TMEM lanes 0-63) over the
//                    same 64 rows of W_up (lanes 64-127); the up warps hand
//                    their values to the gate warps through shared memory
//                    (the drained stages), which store fp16(silu(gate) * up).
// Every wait is bounded; on a timeout the CTA records an error, stops, lets
// issued MMAs finish and frees its TMEM before returning.
#include <cuda.h>

#include "common.cuh"
#include "gemm_fr.h"
#include "gemm_tc.h"

namespace blk {
namespace {

constexpr int kRows = 128;                       // weight rows per CTA (MMA M)
constexpr int kBK = 64;                          // K columns per stage
constexpr int kHalfRows = 64;                    // rows of one weight box
constexpr int kStages = 6;
constexpr int kThreads = 192;                    // producer, MMA, 4 epilogue warps
constexpr int kABytes = kRows * kBK * 2;         // weight tile of a stage: 16 KB
constexpr int kStageBytes = kABytes + kFrMaxRows * kBK * 2;   // + X box of up to 128 rows
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 256 + 1024;
static_assert(kHalfRows * (kFrMaxRows + 1) * 4 <= kStages * kStageBytes, "exchange buffer");

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset), start address in 16-byte units, version 1.
__device__ __forceinline__ uint64_t desc_sw128(const void* p) {
  uint64_t d = (smem_u32(p) & 0x3FFFFu) >> 4;
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// kind::f16 instruction descriptor: D f32, A and B f16, both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
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

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    fr_gemm_kernel(const __grid_constant__ FrGemmParams p) {
  const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int KB = (p.K + kBK - 1) / kBK;
  const int kb0 = (int)((int64_t)split * KB / p.splits);
  const int nkb = (int)((int64_t)(split + 1) * KB / p.splits) - kb0;   // >= 1: splits <= KB

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(tmem_slot)),
        "r"(p.npad)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t tx = (uint32_t)kABytes + (uint32_t)p.npad * kBK * 2;
      // the tile's two 64-row weight boxes of K block kb
      auto load_w = [&](int kb, uint8_t* sa, uint64_t* bar) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const CUtensorMap* m;
          int row;
          if (EPI == kFrGateUp) {
            m = &p.tmW[hf];
            row = tile * kHalfRows;
          } else {
            row = tile * kRows + hf * kHalfRows;
            int seg = 0;   // rows past the last matrix read as zeros
            while (seg < 2 && p.seg_rows[seg + 1] > 0 && row >= p.seg_rows[seg])
              row -= p.seg_rows[seg++];
            m = &p.tmW[seg];
          }
          tma_load_2d(sa + hf * (kHalfRows * 128), m, kb * kBK, row, bar);
        }
      };
      const int pre = nkb < kStages ? nkb : kStages;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], tx);
        load_w(kb0 + i, smem + (size_t)i * kStageBytes, &full[i]);
      }
      griddep_wait();   // X comes from the previous kernel
      griddep_launch();
      for (int i = 0; i < pre; ++i)
        tma_load_2d(smem + (size_t)i * kStageBytes + kABytes, &p.tmX, (kb0 + i) * kBK, 0,
                    &full[i]);
      int issued = pre;
      for (int i = pre; i < nkb; ++i) {
        const int s = i % kStages;
        if (*abort_flag) break;
        if (!mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* sa = smem + (size_t)s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], tx);
        load_w(kb0 + i, sa, &full[s]);
        tma_load_2d(sa + kABytes, &p.tmX, (kb0 + i) * kBK, 0, &full[s]);
        ++issued;
      }
      // copies still in flight land before shared memory goes away
      for (int k = issued > kStages ? issued - kStages : 0; k < issued; ++k)
        mbar_wait(&full[k % kStages], (k / kStages) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc_f16(kRows, p.npad);
      bool ok = true, issued = false;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kStages;
        if (*abort_flag || !mbar_wait(&full[s], (i / kStages) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* sa = smem + (size_t)s * kStageBytes;
        const uint64_t da = desc_sw128(sa), db = desc_sw128(sa + kABytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)   // +32 bytes per K step inside the swizzle atom
          mma_f16(tmem, da + 2 * k, db + 2 * k, id, (i | k) != 0);
        issued = true;
        mma_commit(&empty[s]);
      }
      if (ok) {
        mma_commit(acc_full);
      } else {
        *abort_flag = 1;
        if (issued) {   // let issued MMAs finish before TMEM is freed
          mma_commit(drain);
          mbar_wait(drain, 0, nullptr);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    griddep_wait();   // the previous kernel may still read the output buffer
    griddep_launch();
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int r = q * 32 + lane;             // weight row in the tile
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const int ncols = p.M < p.npad ? p.M : p.npad;   // activation rows with a result
    const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.err));
    if (ok) tc_fence_after();
    if constexpr (EPI == kFrPart) {
      if (ok) {
        const int n = tile * kRows + r;
        float* dst = p.part + (size_t)split * p.M * p.N + n;
        for (int c = 0; c < ncols; c += 32) {
          float v[32];
          tmem_ld32(tl + c, v);
          if (n < p.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c + i < ncols) dst[(size_t)(c + i) * p.N] = v[i];
          }
        }
      }
    } else {
      // up (lanes 64-127) -> shared memory [64][npad + 1] over the drained
      // stages (every copy has landed and been consumed once the
      // accumulator is full); gate (lanes 0-63) reads it back
      float* xch = reinterpret_cast<float*>(smem);
      const int ld = p.npad + 1;   // odd: a warp's 32 rows hit 32 banks
      if (ok && q >= 2) {
        for (int c = 0; c < ncols; c += 32) {
          float v[32];
          tmem_ld32(tl + c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) xch[(r - kHalfRows) * ld + c + i] = v[i];
        }
      }
      named_sync(1, 4 * 32);   // all four epilogue warps, whether or not ok
      if (ok && q < 2) {
        const int j = tile * kHalfRows + r;
        for (int c = 0; c < ncols; c += 32) {
          float v[32];
          tmem_ld32(tl + c, v);
          if (j < p.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c + i < ncols)
                p.out16[(size_t)(c + i) * p.ldo + j] =
                    __float2half_rn(silu(v[i]) * xch[r * ld + c + i]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(p.npad)
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_fr_gemm(FrGemmParams& p, int epi, int num_sms, cudaStream_t s, bool pdl) {
  if (p.M < 1 || p.M > kFrMaxRows || p.N < 1 || p.K < 8 || p.K % 8 || !p.x || !p.w[0])
    return cudaErrorInvalidValue;
  if (epi == kFrPart ? (!p.part || p.max_splits < 1) : (!p.out16 || !p.w[1] || p.ldo < p.N))
    return cudaErrorInvalidValue;
  p.npad = p.M <= 32 ? 32 : (p.M <= 64 ? 64 : 128);
  if (make_tmap_2d(&p.tmX, p.x, p.M, p.K, p.npad)) return cudaErrorInvalidValue;
  const int nw = epi == kFrGateUp ? 2 : 3;
  for (int i = 0; i < nw; ++i) {
    if (!p.w[i]) break;
    const int rows = epi == kFrGateUp ? p.N : p.seg_rows[i];
    if (rows < 1 || make_tmap_2d(&p.tmW[i], p.w[i], rows, p.K, kHalfRows))
      return cudaErrorInvalidValue;
  }
  const int tiles = epi == kFrGateUp ? (p.N + kHalfRows - 1) / kHalfRows : (p.N + kRows - 1) / kRows;
  const int KB = (p.K + kBK - 1) / kBK;
  int S = 1;
  if (epi == kFrPart) {
    S = num_sms / tiles;
    if (S > p.max_splits) S = p.max_splits;
    if (S > KB) S = KB;
    if (S < 1) S = 1;
  }
  p.splits = S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles * S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (epi == kFrGateUp) return cudaLaunchKernelEx(&cfg, fr_gemm_kernel<kFrGateUp>, p);
  return cudaLaunchKernelEx(&cfg, fr_gemm_kernel<kFrPart>, p);
}

cudaError_t configure_fr_gemm_kernels() {
  cudaError_t e = cudaFuncSetAttribute(fr_gemm_kernel<kFrPart>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fr_gemm_kernel<kFrGateUp>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  return e;
}

}  // namespace blk
