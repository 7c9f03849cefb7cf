// Decode-phase projections: one token, so each projection is a matrix-vector
// product bound by the weight bytes streamed from HBM.
//
// Layout of one CTA: 8 consumer warps + 1 producer warp.  The producer's lane
// 0 streams this CTA's weight rows into a ring of shared-memory stages with
// untiled bulk copies (cp.async.bulk, completion on an mbarrier).  It starts
// before griddepcontrol.wait: weights never depend on the previous kernel, so
// under programmatic dependent launch the weight stream of this kernel
// overlaps the tail of the previous one.  Consumers wait for the dependency,
// stage the input vector (RMSNorm applied where the mode needs it) in shared
// memory as fp16, then take the stages: each row's dot product is split over
// `warps_per_row` warps and 32 lanes with 16-byte vectors, fp32 accumulate.
// Per-(row, slice) partial sums land in shared memory and are added in a fixed
// order by the epilogue, so results are deterministic.
#include "common.cuh"
#include "kernels.h"

namespace blk {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;

struct RowBlock {
  const __half* W;
  int row0;
  int n;
  int res_off;
};

// Rows this CTA owns, as one or two contiguous row blocks.
template <int MODE>
__device__ __forceinline__ int cta_blocks(const GemvParams& p, RowBlock* rb) {
  const int b = blockIdx.x, C = gridDim.x;
  if constexpr (MODE == kGemvQKV) {
    const int half = p.D / 2;
    const int hd = b / p.parts, part = b % p.parts;
    const int u0 = part * half / p.parts, u1 = (part + 1) * half / p.parts;
    int seg, local;
    if (hd < p.Hq) {
      seg = 0;
      local = hd;
    } else if (hd < p.Hq + p.Hkv) {
      seg = 1;
      local = hd - p.Hq;
    } else {
      seg = 2;
      local = hd - p.Hq - p.Hkv;
    }
    rb[0] = {p.W[seg], local * p.D + u0, u1 - u0, 0};
    rb[1] = {p.W[seg], local * p.D + half + u0, u1 - u0, u1 - u0};
    return 2;
  } else if constexpr (MODE == kGemvGateUp) {
    const int j0 = (int)((int64_t)b * p.N / C), j1 = (int)((int64_t)(b + 1) * p.N / C);
    rb[0] = {p.W[0], j0, j1 - j0, 0};
    rb[1] = {p.W[1], j0, j1 - j0, j1 - j0};
    return 2;
  } else {
    const int r0 = (int)((int64_t)b * p.N / C), r1 = (int)((int64_t)(b + 1) * p.N / C);
    rb[0] = {p.W[0], r0, r1 - r0, 0};
    return 1;
  }
}

template <int MODE>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_stream_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int SB = p.stage_bytes, NS = p.n_stages, K = p.K;
  unsigned char* ring = smem;
  __half* xs = reinterpret_cast<__half*>(smem + (size_t)NS * SB);
  float* part = reinterpret_cast<float*>(xs + ((K + 7) & ~7));
  float* red = part + ((p.max_rows * p.warps_per_row + 3) & ~3);  // [32]
  int* abort_flag = reinterpret_cast<int*>(red + 32);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 36);   // [NS], 16B aligned
  uint64_t* empty = full + NS;                              // [NS]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  RowBlock rb[2];
  const int nb = cta_blocks<MODE>(p, rb);
  const int CR = p.rows_per_chunk;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    int c = 0;
    bool ok = true;
    for (int b = 0; b < nb && ok; ++b) {
      for (int r = 0; r < rb[b].n; r += CR) {
        const int rows = min(CR, rb[b].n - r);
        const uint32_t bytes = (uint32_t)rows * (uint32_t)K * 2u;
        const int s = c % NS;
        if (c >= NS && !mbar_wait(&empty[s], ((c / NS) - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(ring + (size_t)s * SB, rb[b].W + (size_t)(rb[b].row0 + r) * K,
                 bytes, &full[s]);
        ++c;
      }
    }
    if (!ok) {
      // Let the copies already issued land before the CTA's memory goes away.
      for (int k = max(0, c - NS); k < c; ++k)
        mbar_wait(&full[k % NS], (k / NS) & 1, nullptr);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int tid = threadIdx.x;  // < 256
  constexpr int kC = kConsumerWarps * 32;
  griddep_wait();
  griddep_launch();

  if constexpr (MODE == kGemvQKV) {
    if (blockIdx.x == 0)
      for (int i = tid; i < p.n_counters; i += kC) p.counters[i] = 0u;
  }

  // Stage the input vector (fp16) in shared memory.
  if constexpr (MODE == kGemvQKV || MODE == kGemvGateUp) {
    float ss = 0.f;
    for (int i = tid; i < K; i += kC) {
      const float v = (MODE == kGemvQKV) ? __half2float(p.x16[i]) : p.x32[i];
      ss += v * v;
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    named_sync(1, kC);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += red[w];
    const float rstd = rsqrtf(tot / (float)K + p.eps);
    for (int i = tid; i < K; i += kC) {
      const float v = (MODE == kGemvQKV) ? __half2float(p.x16[i]) : p.x32[i];
      xs[i] = __float2half_rn(v * rstd * __half2float(p.gain[i]));
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(p.x16);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    for (int i = tid; i < K / 8; i += kC) dst[i] = src[i];
  }
  named_sync(1, kC);

  const int WPR = p.warps_per_row;
  const int nv = K / 8;
  const int my_row = warp / WPR, my_slice = warp % WPR;
  const int v0 = my_slice * nv / WPR, v1 = (my_slice + 1) * nv / WPR;
  const uint4* x4 = reinterpret_cast<const uint4*>(xs);
  int c = 0;
  bool ok = true;
  for (int b = 0; b < nb && ok; ++b) {
    for (int r = 0; r < rb[b].n; r += CR) {
      const int rows = min(CR, rb[b].n - r);
      const int s = c % NS;
      if (!mbar_wait(&full[s], (c / NS) & 1, p.err)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      if (my_row < rows) {
        const uint4* w4 = reinterpret_cast<const uint4*>(ring + (size_t)s * SB +
                                                         (size_t)my_row * K * 2);
        float a0 = 0.f, a1 = 0.f;
        int v = v0 + lane;
        for (; v + 32 < v1; v += 64) {
          float fw[8], fx[8], gw[8], gx[8];
          h8_to_f32(w4[v], fw);
          h8_to_f32(x4[v], fx);
          h8_to_f32(w4[v + 32], gw);
          h8_to_f32(x4[v + 32], gx);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            a0 = fmaf(fw[i], fx[i], a0);
            a1 = fmaf(gw[i], gx[i], a1);
          }
        }
        if (v < v1) {
          float fw[8], fx[8];
          h8_to_f32(w4[v], fw);
          h8_to_f32(x4[v], fx);
#pragma unroll
          for (int i = 0; i < 8; ++i) a0 = fmaf(fw[i], fx[i], a0);
        }
        const float dot = warp_sum(a0 + a1);
        if (lane == 0) part[(rb[b].res_off + r + my_row) * WPR + my_slice] = dot;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      ++c;
    }
  }
  // Every consumer warp reaches this barrier, also after a timed-out wait.
  named_sync(1, kC);
  if (*abort_flag) return;

  auto val = [&](int row) {
    float a = 0.f;
    for (int k = 0; k < WPR; ++k) a += part[row * WPR + k];
    return a;
  };

  if constexpr (MODE == kGemvQKV) {
    const int half = p.D / 2;
    const int hd = blockIdx.x / p.parts, prt = blockIdx.x % p.parts;
    const int u0 = prt * half / p.parts;
    const int n = rb[0].n;
    const int64_t pos = p.pos[0];
    for (int k = tid; k < n; k += kC) {
      const int i = u0 + k;
      float lo = val(k), hi = val(n + k);
      if (hd < p.Hq) {
        if (p.bias[0]) {
          lo += __half2float(p.bias[0][hd * p.D + i]);
          hi += __half2float(p.bias[0][hd * p.D + half + i]);
        }
        const float2 cs = rope_cs(p.rope, p.rope_len, half, pos, i, p.err);
        p.q32[hd * p.D + i] = lo * cs.x - hi * cs.y;
        p.q32[hd * p.D + half + i] = hi * cs.x + lo * cs.y;
      } else if (hd < p.Hq + p.Hkv) {
        const int g = hd - p.Hq;
        if (p.bias[1]) {
          lo += __half2float(p.bias[1][g * p.D + i]);
          hi += __half2float(p.bias[1][g * p.D + half + i]);
        }
        const float2 cs = rope_cs(p.rope, p.rope_len, half, pos, i, p.err);
        const __half a = __float2half_rn(lo * cs.x - hi * cs.y);
        const __half bb = __float2half_rn(hi * cs.x + lo * cs.y);
        __half* dst = p.kc + ((size_t)g * p.max_ctx + p.slot) * p.D;
        dst[i] = a;
        dst[half + i] = bb;
        if (p.k_new) {
          p.k_new[g * p.D + i] = a;
          p.k_new[g * p.D + half + i] = bb;
        }
      } else {
        const int g = hd - p.Hq - p.Hkv;
        if (p.bias[2]) {
          lo += __half2float(p.bias[2][g * p.D + i]);
          hi += __half2float(p.bias[2][g * p.D + half + i]);
        }
        const __half a = __float2half_rn(lo), bb = __float2half_rn(hi);
        __half* dst = p.vc + ((size_t)g * p.max_ctx + p.slot) * p.D;
        dst[i] = a;
        dst[half + i] = bb;
        if (p.v_new) {
          p.v_new[g * p.D + i] = a;
          p.v_new[g * p.D + half + i] = bb;
        }
      }
    }
  } else if constexpr (MODE == kGemvGateUp) {
    const int n = rb[0].n, j0 = rb[0].row0;
    for (int k = tid; k < n; k += kC)
      p.out16[j0 + k] = __float2half_rn(silu(val(k)) * val(n + k));
  } else if constexpr (MODE == kGemvO) {
    const int n = rb[0].n, r0 = rb[0].row0;
    for (int k = tid; k < n; k += kC)
      p.out32[r0 + k] = val(k) + __half2float(p.res16[r0 + k]);
  } else {
    const int n = rb[0].n, r0 = rb[0].row0;
    for (int k = tid; k < n; k += kC)
      p.out16[r0 + k] = __float2half_rn(val(k) + p.res32[r0 + k]);
  }
}

// ---------------------------------------------------------------- host side

static void gemv_geometry(GemvParams& p, int mode, int grid) {
  const int row_bytes = p.K * 2;
  int cr = 8;
  while (cr > 1 && cr * row_bytes > 24 * 1024) cr >>= 1;
  p.rows_per_chunk = cr;
  p.warps_per_row = kConsumerWarps / cr;
  p.stage_bytes = cr * row_bytes;
  int ns = (88 * 1024) / p.stage_bytes;
  p.n_stages = ns < 2 ? 2 : (ns > 8 ? 8 : ns);
  int max_rows;
  if (mode == kGemvQKV) {
    const int half = p.D / 2;
    max_rows = 2 * ((half + p.parts - 1) / p.parts);
  } else if (mode == kGemvGateUp) {
    max_rows = 2 * ((p.N + grid - 1) / grid);
  } else {
    max_rows = (p.N + grid - 1) / grid;
  }
  p.max_rows = max_rows;
}

static size_t gemv_smem(const GemvParams& p) {
  return (size_t)p.n_stages * p.stage_bytes + (size_t)((p.K + 7) & ~7) * 2 +
         (size_t)((p.max_rows * p.warps_per_row + 3) & ~3) * 4 + 36 * 4 +
         (size_t)2 * p.n_stages * 8;
}

int gemv_grid(const GemvParams& p, int mode, int num_sms) {
  if (mode == kGemvQKV) {
    const int heads = p.Hq + 2 * p.Hkv;
    return heads * p.parts;
  }
  const int rows = p.N;
  return rows < num_sms ? rows : num_sms;
}

template <int MODE>
static cudaError_t launch_mode(const GemvParams& p, int grid, cudaStream_t s,
                               bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = gemv_smem(p);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_stream_kernel<MODE>, p);
}

cudaError_t launch_gemv(GemvParams p, int mode, int grid, cudaStream_t s,
                        bool pdl) {
  gemv_geometry(p, mode, grid);
  switch (mode) {
    case kGemvQKV: return launch_mode<kGemvQKV>(p, grid, s, pdl);
    case kGemvO: return launch_mode<kGemvO>(p, grid, s, pdl);
    case kGemvGateUp: return launch_mode<kGemvGateUp>(p, grid, s, pdl);
    default: return launch_mode<kGemvDown>(p, grid, s, pdl);
  }
}

cudaError_t configure_gemv_kernels() {
  const int limit = 227 * 1024;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemv_stream_kernel<kGemvQKV>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, limit)))
    return e;
  if ((e = cudaFuncSetAttribute(gemv_stream_kernel<kGemvO>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, limit)))
    return e;
  if ((e = cudaFuncSetAttribute(gemv_stream_kernel<kGemvGateUp>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, limit)))
    return e;
  return cudaFuncSetAttribute(gemv_stream_kernel<kGemvDown>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
}

}  // namespace blk
