// Decode: one token through a stack of decoder blocks in ONE persistent,
// cooperative kernel launch.
//
// At one token every projection is a matrix-vector product: the step is
// bound by the bytes of the weights (93.6 MB per 1.5B-shaped layer) and of
// the KV history.  Those bytes never depend on the token being decoded, so
// each CTA (one per SM) has a producer lane that streams, in consumption
// order, every weight row block and every KV-history tile the CTA will use —
// across phase and layer boundaries — into a 4 x 48 KB shared-memory ring
// (untiled bulk copies for weight rows; 128B-swizzled tensor copies for K/V
// tiles).  Twelve consumer warps run the phases of each layer and meet at a
// grid-wide barrier between phases; while they wait, the producer keeps
// filling the ring, so HBM stays busy through the barriers.
//
// Phases of one layer (the block of the TopOp paper, Listing 2, at T = 1):
//   QKV   RMSNorm(x) staged in shared memory; rows of wq|wk|wv in RoPE pairs
//         (i, i + D/2); epilogue: bias, RoPE, q (fp32) to the workspace, K/V
//         to cache slot cache_len and to k_new / v_new.
//   ATTN  CTA (kv head g, split s) covers slots [j0, j1) of [0, cache_len];
//         4 warps run mma.sync m16n8k16 (rows = the G query heads of the
//         group, padded to 16) over 64-slot tiles: S = Q K^T, online softmax
//         in base 2, O += P V; the warps' states are merged and one partial
//         (acc, max, sum) per query head is written.
//   COMB  every CTA merges all splits for a slice of (head, d) pairs -> attn.
//   O     rows of wo; epilogue h = acc + x (fp32).
//   GU    RMSNorm(h) staged; matching rows of w_gate and w_up; epilogue
//         silu(gate) * up (fp16).
//   DOWN  rows of w_down; epilogue out = acc + h (fp16) = next layer's input.
// Dot products are split over warps and lanes with 16-byte vectors and fp32
// accumulation; per-(row, slice) partials are added in a fixed order, so the
// result does not depend on timing.
//
// Every wait (ring mbarriers, grid barrier) is bounded; on a timeout the
// kernel records an error, stops, lets its issued copies land and returns.
#include "common.cuh"
#include "decode_persistent.h"

namespace blk {
namespace {

// 12 consumer warps + 1 producer warp: 13 warps, so no SM sub-partition holds
// more than 4 and each thread may use up to 128 registers without spilling.
constexpr int kCW = 12;                 // consumer warps
constexpr int kCT = kCW * 32;           // consumer threads
constexpr int kThreads = kCT + 32;      // + one producer warp
constexpr int kStageBytes = 48 * 1024;
constexpr int kStages = 4;
constexpr int kAttnWarps = 4;           // 4 x 16 slots = one 64-slot tile
constexpr int kSlots = 64;
constexpr int kGroupRows = 15;          // weight rows per mma tile (of 16)
constexpr int kKc = 1536;               // weight columns per ring stage
constexpr int kRowStride = (kKc + 8) * 2;  // bytes per staged row: 16-byte pad
                                           // keeps ldmatrix free of conflicts
constexpr int kPartFloats = 2048;       // [row group][warp][16] partial sums
constexpr int kQStride = 136;           // Q tile row stride in halves (padded)
static_assert(kGroupRows * kRowStride <= kStageBytes, "stage too small");

constexpr int kXsOff = kStages * kStageBytes;
constexpr int kPartOff = kXsOff + kDecMaxVec * 2;
constexpr int kQOff = kPartOff;         // the Q tile reuses the partials area
constexpr int kBarOff = kPartOff + kPartFloats * 4;
constexpr int kResRows = 150;           // hidden rows per CTA (o_proj / down)
constexpr int kResOff = kBarOff + 256;  // x and h slices of this CTA's rows
constexpr int kSmemUsed = kResOff + 2 * kResRows * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + alignment slack

enum Phase { kPhQKV = 0, kPhAttn = 1, kPhComb = 2, kPhO = 3, kPhGU = 4, kPhDown = 5 };
constexpr int kPhases = 6;

// ------------------------------------------------------------ small PTX
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
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

// Address of the 16-byte chunk `ch` (8 halves) of row `r` in a 64-row tile
// stored as 128-byte-swizzled half tiles of 64 columns (8 KB each).
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int ch) {
  const int half = ch >> 3, c = ch & 7;
  return base + half * 8192 + r * 128 + ((c ^ (r & 7)) << 4);
}

// ------------------------------------------------------------ schedule
__device__ __forceinline__ const __half* layer_input(const DecodeParams& p, int l) {
  return l == 0 ? p.x_in : ((l - 1) & 1 ? p.xbuf1 : p.xbuf0);
}
__device__ __forceinline__ __half* layer_output(const DecodeParams& p, int l) {
  return l == p.n_layers - 1 ? p.out : (l & 1 ? p.xbuf1 : p.xbuf0);
}

// The weight rows one CTA owns in a projection phase, as a list indexed by
// q in [0, nrows):
//   QKV  q <  units: row i of head hd (pair unit u = u0 + q, i = u % (D/2))
//        q >= units: its partner row i + D/2
//   GU   q <  units: W_gate row j0 + q;  q >= units: W_up row j0 + q - units
//   O, DOWN  row r0 + q
struct PhaseRows {
  int nrows, units, K, first, ncol;
};

__device__ __forceinline__ PhaseRows phase_rows(const DecodeParams& p, int ph) {
  const int b = blockIdx.x, G = gridDim.x;
  PhaseRows r;
  int total;
  if (ph == kPhQKV) { total = (p.Hq + 2 * p.Hkv) * (p.D / 2); r.K = p.H; }
  else if (ph == kPhGU) { total = p.I; r.K = p.H; }
  else { total = p.H; r.K = ph == kPhO ? p.Hq * p.D : p.I; }
  r.first = (int)((int64_t)b * total / G);
  r.units = (int)((int64_t)(b + 1) * total / G) - r.first;
  r.nrows = (ph == kPhQKV || ph == kPhGU) ? 2 * r.units : r.units;
  r.ncol = (r.K + kKc - 1) / kKc;
  return r;
}

__device__ __forceinline__ const __half* row_ptr(const DecodeParams& p, const DecLayer& Ly,
                                                 int ph, const PhaseRows& r, int q) {
  if (ph == kPhQKV) {
    const int half = p.D / 2;
    const bool hi = q >= r.units;
    const int u = r.first + (hi ? q - r.units : q);
    const int hd = u / half, i = u % half + (hi ? half : 0);
    const __half* W;
    int local;
    if (hd < p.Hq) { W = Ly.wq; local = hd; }
    else if (hd < p.Hq + p.Hkv) { W = Ly.wk; local = hd - p.Hq; }
    else { W = Ly.wv; local = hd - p.Hq - p.Hkv; }
    return W + (size_t)(local * p.D + i) * r.K;
  }
  if (ph == kPhGU) {
    return q < r.units ? Ly.wg + (size_t)(r.first + q) * r.K
                       : Ly.wu + (size_t)(r.first + q - r.units) * r.K;
  }
  return (ph == kPhO ? Ly.wo : Ly.wd) + (size_t)(r.first + q) * r.K;
}

struct AttnRange {
  bool active;
  int g, s;
  int64_t j0, j1;  // slots [j0, j1) of [0, cache_len + 1)
  int chunks;
};

__device__ __forceinline__ AttnRange attn_range(const DecodeParams& p) {
  AttnRange a;
  const int b = blockIdx.x;
  a.active = b < p.Hkv * p.S;
  a.g = b / p.S;
  a.s = b % p.S;
  const int64_t n = p.cache_len + 1;
  a.j0 = a.active ? (int64_t)a.s * n / p.S : 0;
  a.j1 = a.active ? (int64_t)(a.s + 1) * n / p.S : 0;
  a.chunks = (int)((a.j1 - a.j0 + kSlots - 1) / kSlots);
  return a;
}

// ------------------------------------------------------------ grid barrier
struct Sync {
  unsigned* counter;
  int* err;
  volatile int* abort_flag;
};

// All consumer threads of every CTA call arrive() after their writes of a
// phase; wait(k) returns once all CTAs arrived at barrier k (0-based).
__device__ __forceinline__ void grid_arrive(const Sync& s) {
  named_sync(1, kCT);
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(s.counter, 1u);
  }
}

__device__ __forceinline__ bool grid_wait(const Sync& s, int k) {
  if (threadIdx.x == 0 && !*s.abort_flag) {
    const unsigned target = (unsigned)(k + 1) * gridDim.x;
    if (ld_acquire(s.counter) < target) {
      const uint64_t t0 = global_ns();
      while (ld_acquire(s.counter) < target) {
        if (global_ns() - t0 > kWaitLimitNs) {
          set_error(s.err, kDevTimeout);
          *s.abort_flag = 1;
          break;
        }
      }
    }
    __threadfence();
  }
  named_sync(1, kCT);
  return !*s.abort_flag;
}

// ------------------------------------------------------------ staging
// Inputs written by other CTAs in the previous phase are read with ld.global.cg
// (L2, never a stale L1 line).  Every thread issues all its loads first, so a
// staging step costs one L2 round trip.
constexpr int kMaxV16 = (kDecMaxVec / 8 + kCT - 1) / kCT;  // uint4 per thread (fp16)
constexpr int kMaxV32 = (kDecMaxVec / 4 + kCT - 1) / kCT;  // float4 per thread (fp32)

// xs[i] = fp16(x[i] * rsqrt(mean(x^2) + eps) * g[i]) for fp16 x.
// Also copies x[cap_lo, cap_hi) (raw) to cap[] for a later residual.
__device__ void stage_rmsnorm16(const __half* x, const __half* g, int K, float eps, __half* xs,
                                float* red, int cap_lo, int cap_hi, float* cap) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nv = K / 8;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  uint4 v[kMaxV16];
#pragma unroll
  for (int k = 0; k < kMaxV16; ++k) {
    const int i = tid + k * kCT;
    v[k] = i < nv ? __ldcg(x4 + i) : make_uint4(0, 0, 0, 0);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxV16; ++k) {
    float f[8];
    h8_to_f32(v[k], f);
    const int i0 = 8 * (tid + k * kCT);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ss += f[e] * f[e];
      if (i0 + e >= cap_lo && i0 + e < cap_hi) cap[i0 + e - cap_lo] = f[e];
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  named_sync(1, kCT);
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kCW; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)K + eps);
  const uint4* g4 = reinterpret_cast<const uint4*>(g);
#pragma unroll
  for (int k = 0; k < kMaxV16; ++k) {
    const int i = tid + k * kCT;
    if (i < nv) {
      float f[8], gf[8];
      h8_to_f32(v[k], f);
      h8_to_f32(__ldg(g4 + i), gf);
      uint4 o;
      __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        oh[e] = __floats2half2_rn(f[2 * e] * r * gf[2 * e], f[2 * e + 1] * r * gf[2 * e + 1]);
      reinterpret_cast<uint4*>(xs)[i] = o;
    }
  }
  named_sync(1, kCT);
}

// Same for fp32 x (the residual stream h).
__device__ void stage_rmsnorm32(const float* x, const __half* g, int K, float eps, __half* xs,
                                float* red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nv = K / 4;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  float4 v[kMaxV32];
#pragma unroll
  for (int k = 0; k < kMaxV32; ++k) {
    const int i = tid + k * kCT;
    v[k] = i < nv ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxV32; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  named_sync(1, kCT);
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kCW; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)K + eps);
  const uint2* g2 = reinterpret_cast<const uint2*>(g);
#pragma unroll
  for (int k = 0; k < kMaxV32; ++k) {
    const int i = tid + k * kCT;
    if (i < nv) {
      const uint2 graw = __ldg(g2 + i);
      const float2 ga = __half22float2(*reinterpret_cast<const __half2*>(&graw.x));
      const float2 gb = __half22float2(*reinterpret_cast<const __half2*>(&graw.y));
      uint2 o;
      *reinterpret_cast<__half2*>(&o.x) = __floats2half2_rn(v[k].x * r * ga.x, v[k].y * r * ga.y);
      *reinterpret_cast<__half2*>(&o.y) = __floats2half2_rn(v[k].z * r * gb.x, v[k].w * r * gb.y);
      reinterpret_cast<uint2*>(xs)[i] = o;
    }
  }
  named_sync(1, kCT);
}

__device__ void stage_copy(const __half* src, int K, __half* xs) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(xs);
  const int nv = K / 8;
  uint4 v[kMaxV16];
#pragma unroll
  for (int k = 0; k < kMaxV16; ++k) {
    const int i = threadIdx.x + k * kCT;
    if (i < nv) v[k] = __ldcg(s4 + i);
  }
#pragma unroll
  for (int k = 0; k < kMaxV16; ++k) {
    const int i = threadIdx.x + k * kCT;
    if (i < nv) d4[i] = v[k];
  }
  named_sync(1, kCT);
}

// o_proj input when the attention used few splits: xs[h*D + d] = attention
// output of query head h, merged here from the S split partials (acc, max,
// sum) instead of in a separate phase.  One thread per 4 consecutive d.
template <int D>
__device__ void stage_combine(const DecodeParams& p, __half* xs) {
  constexpr int kMaxS = 32;
  const int n4 = p.Hq * D / 4;
  for (int c = threadIdx.x; c < n4; c += kCT) {
    const int hq = (4 * c) / D, d = (4 * c) % D;
    const float* base = p.part + (size_t)hq * p.S * (D + 4);
    float2 ml[kMaxS];   // (max, sum) of every split, loaded first
#pragma unroll
    for (int s = 0; s < kMaxS; ++s)
      ml[s] = s < p.S ? __ldcg(reinterpret_cast<const float2*>(base + (size_t)s * (D + 4) + D))
                      : make_float2(-INFINITY, 0.f);
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxS; ++s) M = fmaxf(M, ml[s].x);
    float Ls = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s0 = 0; s0 < kMaxS; s0 += 8) {   // accumulators in batches of 8 loads
      if (s0 >= p.S) break;
      float4 a[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        a[k] = s0 + k < p.S
                   ? __ldcg(reinterpret_cast<const float4*>(base + (size_t)(s0 + k) * (D + 4) + d))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float w = ml[s0 + k].x == -INFINITY ? 0.f : exp2f(ml[s0 + k].x - M);
        Ls += ml[s0 + k].y * w;
        O.x += a[k].x * w; O.y += a[k].y * w; O.z += a[k].z * w; O.w += a[k].w * w;
      }
    }
    const float inv = 1.f / Ls;
    __half2* dst = reinterpret_cast<__half2*>(xs + hq * D + d);
    dst[0] = __floats2half2_rn(O.x * inv, O.y * inv);
    dst[1] = __floats2half2_rn(O.z * inv, O.w * inv);
  }
  named_sync(1, kCT);
}

// Position in this CTA's stream of ring chunks: layer l, phase ph, and
// within the phase either the K/V tile c or the (row group g0, column chunk
// kc) of the phase's weight rows.
struct Cursor {
  int l, ph, c, g0, kc;
  PhaseRows R;
};

// Settles on the first chunk at or after (l, ph); false past the last layer.
__device__ bool cursor_begin(Cursor& cu, const DecodeParams& p, const AttnRange& ar) {
  for (; cu.l < p.n_layers; ++cu.l, cu.ph = 0) {
    for (; cu.ph < kPhases; ++cu.ph) {
      if (cu.ph == kPhComb) continue;
      if (cu.ph == kPhAttn) {
        if (ar.chunks > 0) { cu.c = 0; return true; }
        continue;
      }
      cu.R = phase_rows(p, cu.ph);
      if (cu.R.nrows > 0) { cu.g0 = 0; cu.kc = 0; return true; }
    }
  }
  return false;
}

__device__ bool cursor_next(Cursor& cu, const DecodeParams& p, const AttnRange& ar) {
  if (cu.ph == kPhAttn) {
    if (++cu.c < ar.chunks) return true;
  } else {
    if (++cu.kc < cu.R.ncol) return true;
    cu.kc = 0;
    cu.g0 += kGroupRows;
    if (cu.g0 < cu.R.nrows) return true;
  }
  ++cu.ph;
  return cursor_begin(cu, p, ar);
}

// Optional timeline: thread 0 of every CTA records %globaltimer when a phase
// starts (after its barrier) and when its work is done.
__device__ __forceinline__ void trace_point(const DecodeParams& p, int l, int ph, int k) {
  if (p.trace && threadIdx.x == 0) {
    const size_t i = (((size_t)blockIdx.x * p.n_layers + l) * kPhases + ph) * 2 + k;
    if (i < p.trace_len) p.trace[i] = global_ns();
  }
}

// ------------------------------------------------------------ the kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_persistent_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  __half* xs = reinterpret_cast<__half*>(smem + kXsOff);
  float* part = reinterpret_cast<float*>(smem + kPartOff);
  __half* qtile = reinterpret_cast<__half*>(smem + kQOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  float* red = reinterpret_cast<float*>(empty + kStages);        // [16]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 16);
  float* xres = reinterpret_cast<float*>(smem + kResOff);       // x[r0 + k]
  float* hres = xres + kResRows;                                // h[r0 + k]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const AttnRange ar = attn_range(p);
  const int G = p.Hq / p.Hkv;
  constexpr int kv_tile_bytes = kSlots * D * 2;  // one of K or V for a 64-slot tile

  // ================================================================ producer
  // Lane 0 walks this CTA's chunk stream and loads each chunk into the next
  // free ring stage.
  if (warp == kCW) {
    if (lane != 0) return;
    auto chunk_bytes = [&](const Cursor& cu) -> uint32_t {
      if (cu.ph == kPhAttn) return 2u * kv_tile_bytes;
      const int nr = min(kGroupRows, cu.R.nrows - cu.g0);
      return (uint32_t)nr * (uint32_t)min(kKc, cu.R.K - cu.kc * kKc) * 2u;
    };
    auto kv_row = [&](const Cursor& cu) {
      return (int)(ar.g * p.max_ctx + ar.j0 + (int64_t)cu.c * kSlots);
    };
    auto load = [&](const Cursor& cu, uint8_t* st, uint64_t* bar) {
      if (cu.ph == kPhAttn) {
        const int y = kv_row(cu);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_2d(st + h * 8192, &p.tm_k[cu.l], h * 64, y, bar);
          tma_load_2d(st + kv_tile_bytes + h * 8192, &p.tm_v[cu.l], h * 64, y, bar);
        }
        return;
      }
      const int nr = min(kGroupRows, cu.R.nrows - cu.g0);
      const uint32_t rb = (uint32_t)min(kKc, cu.R.K - cu.kc * kKc) * 2u;
      for (int r = 0; r < nr; ++r)
        bulk_g2s(st + r * kRowStride,
                 row_ptr(p, p.layer[cu.l], cu.ph, cu.R, cu.g0 + r) + cu.kc * kKc, rb, bar);
    };
    Cursor rc = {0, 0, 0, 0, 0, {}};
    bool more = cursor_begin(rc, p, ar);
    int it = 0;   // chunks issued to the ring
    bool ok = true;
    while (more && ok) {
      const int s = it % kStages;
      if (it >= kStages) {
        const uint32_t par = ((it / kStages) - 1) & 1;
        uint64_t t0 = 0;
        while (!mbar_test(&empty[s], par)) {
          if (*abort_flag) { ok = false; break; }
          if (t0 == 0) t0 = global_ns();
          else if (global_ns() - t0 > kWaitLimitNs) {
            set_error(p.err, kDevTimeout);
            *abort_flag = 1;
            ok = false;
            break;
          }
        }
        if (!ok) break;
      }
      mbar_arrive_expect_tx(&full[s], chunk_bytes(rc));
      load(rc, ring + (size_t)s * kStageBytes, &full[s]);
      ++it;
      more = cursor_next(rc, p, ar);
    }
    // Copies still in flight must land before the CTA's shared memory goes away.
    for (int k = max(0, it - kStages); k < it; ++k)
      mbar_wait(&full[k % kStages], (k / kStages) & 1, nullptr);
    return;
  }

  // ================================================================ consumers
  const Sync sync{p.barrier, p.err, abort_flag};
  int it = 0;          // ring position, in step with the producer
  int bar = 0;         // grid barriers passed
  auto take = [&](int& s) -> bool {   // wait for the next ring stage
    s = it % kStages;
    if (*abort_flag) return false;
    if (!mbar_wait(&full[s], (it / kStages) & 1, p.err)) {
      *abort_flag = 1;
      return false;
    }
    return true;
  };
  auto give = [&](int s) {            // release a ring stage
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ++it;
  };
  const int64_t L = p.cache_len;
  const int64_t pos = p.pos[0];
  const int half = D / 2;

  for (int l = 0; l < p.n_layers; ++l) {
    const DecLayer& Ly = p.layer[l];
    const __half* x_l = layer_input(p, l);
    for (int ph = 0; ph < kPhases; ++ph) {
      if (ph == kPhComb && p.fold) continue;   // merged into the o_proj staging
      // wait for the producers of this phase's input
      if (!(l == 0 && ph == kPhQKV)) {
        if (!grid_wait(sync, bar++)) return;
      }
      trace_point(p, l, ph, 0);

      if (ph == kPhAttn) {
        // ---------------------------------------------------- attention
        // Q tile [16 rows][D]: the G query heads of kv head g, scaled.
        if (warp < kAttnWarps) {
          // 16 x D values = up to 4 float4 per thread, all loads issued first
          constexpr int kAT = kAttnWarps * 32;
          const int n4 = 16 * D / 4;
          const float4* q4 = reinterpret_cast<const float4*>(p.q32 + (size_t)ar.g * G * D);
          float4 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = tid + k * kAT, r = (4 * i) / D;
            v[k] = (i < n4 && ar.active && r < G) ? __ldcg(q4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = tid + k * kAT;
            if (i < n4) {
              const int r = (4 * i) / D, d = (4 * i) % D;
              const float sc = p.scale_log2;
              __half2* dst = reinterpret_cast<__half2*>(qtile + r * kQStride + d);
              dst[0] = __floats2half2_rn(v[k].x * sc, v[k].y * sc);
              dst[1] = __floats2half2_rn(v[k].z * sc, v[k].w * sc);
            }
          }
          named_sync(2, kAttnWarps * 32);
        }
        const int grp = lane >> 2, tig = lane & 3;
        float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
        float O[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
        const uint32_t qbase = smem_u32(qtile);
        const __half* kc_head = Ly.kc + (size_t)ar.g * p.max_ctx * D;
        const __half* vc_head = Ly.vc + (size_t)ar.g * p.max_ctx * D;
        for (int c = 0; c < ar.chunks; ++c) {
          int s;
          if (!take(s)) break;
          if (warp < kAttnWarps) {
            uint8_t* st = ring + (size_t)s * kStageBytes;
            const uint32_t kb = smem_u32(st), vb = kb + kv_tile_bytes;
            const int64_t cs = ar.j0 + (int64_t)c * kSlots;
            const int nval = (int)min((int64_t)kSlots, ar.j1 - cs);
            const int r0 = warp * 16;
            if (r0 < nval) {
              // rows of this warp: the new token's K/V (written by the QKV
              // phase after the tile was fetched) and zero past the range
              const int cpr = D / 8;  // 16-byte chunks per row
#pragma unroll
              for (int idx = lane; idx < 16 * cpr; idx += 32) {
                const int r = r0 + idx / cpr, ch = idx % cpr;
                const int64_t j = cs + r;
                uint4 kv_k, kv_v;
                bool write = false;
                if (j == L) {
                  kv_k = __ldcg(reinterpret_cast<const uint4*>(kc_head + L * D) + ch);
                  kv_v = __ldcg(reinterpret_cast<const uint4*>(vc_head + L * D) + ch);
                  write = true;
                } else if (r >= nval) {
                  kv_k = kv_v = make_uint4(0, 0, 0, 0);
                  write = true;
                }
                if (write) {
                  *reinterpret_cast<uint4*>(st + (tile_addr(kb, r, ch) - kb)) = kv_k;
                  *reinterpret_cast<uint4*>(st + (tile_addr(vb, r, ch) - kb)) = kv_v;
                }
              }
              __syncwarp();
              // S = Q K^T for 16 slots (two n-tiles of 8)
              float S[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t a[4], bk[4];
                {
                  const int m = lane >> 3, rr = (m & 1) * 8 + (lane & 7);
                  const int col = ks * 16 + (m >> 1) * 8;
                  ldsm_x4(qbase + (rr * kQStride + col) * 2, a);
                }
                {
                  const int m = lane >> 3;
                  const int r = r0 + (m >> 1) * 8 + (lane & 7);
                  const int ch = ks * 2 + (m & 1);
                  ldsm_x4(tile_addr(kb, r, ch), bk);
                }
                mma16816(S[0], a, bk[0], bk[1]);
                mma16816(S[1], a, bk[2], bk[3]);
              }
              // online softmax (rows grp and grp + 8 = query heads)
              float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int r = r0 + nt * 8 + 2 * tig + (e & 1);
                  if (r >= nval) S[nt][e] = -INFINITY;
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
              // A fragment of P: (row grp, slots 0-7) (row grp+8, 0-7) (grp, 8-15) (grp+8, 8-15)
              const uint32_t afr[4] = {pa[0], pa[1], pa[2], pa[3]};
#pragma unroll
              for (int dn = 0; dn < D / 8; ++dn) {
                O[dn][0] *= corr[0]; O[dn][1] *= corr[0];
                O[dn][2] *= corr[1]; O[dn][3] *= corr[1];
              }
#pragma unroll
              for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t bv[4];
                const int m = lane >> 3;
                const int r = r0 + (m & 1) * 8 + (lane & 7);
                const int ch = dp * 2 + (m >> 1);
                ldsm_x4_t(tile_addr(vb, r, ch), bv);
                mma16816(O[2 * dp], afr, bv[0], bv[1]);
                mma16816(O[2 * dp + 1], afr, bv[2], bv[3]);
              }
            }
          }
          give(s);
        }
        // every consumer thread passes this barrier, also after an abort
        named_sync(1, kCT);
        if (*abort_flag) return;
        // merge the attention warps' states; write the split's partials
        if (warp < kAttnWarps) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            l_r[h2] += __shfl_xor_sync(0xffffffffu, l_r[h2], 1);
            l_r[h2] += __shfl_xor_sync(0xffffffffu, l_r[h2], 2);
          }
          float* sm_m = reinterpret_cast<float*>(xs);   // [16]
          float* sm_l = sm_m + 16;                      // [16]
          float* sm_o = sm_l + 16;                      // [16][D]
          for (int w = 0; w < kAttnWarps; ++w) {
            if (warp == w) {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const int row = grp + 8 * h2;
                float a = 0.f, bsc = 1.f, Mx = m_r[h2];
                if (w > 0) {
                  const float mo = sm_m[row];
                  Mx = fmaxf(mo, m_r[h2]);
                  a = (Mx == -INFINITY) ? 0.f : exp2f(mo - Mx);
                  bsc = (Mx == -INFINITY) ? 0.f : exp2f(m_r[h2] - Mx);
                }
#pragma unroll
                for (int dn = 0; dn < D / 8; ++dn) {
                  const int col = dn * 8 + 2 * tig;
                  float o0 = O[dn][2 * h2] * bsc, o1 = O[dn][2 * h2 + 1] * bsc;
                  if (w > 0) {
                    o0 += sm_o[row * D + col] * a;
                    o1 += sm_o[row * D + col + 1] * a;
                  }
                  sm_o[row * D + col] = o0;
                  sm_o[row * D + col + 1] = o1;
                }
                __syncwarp();
                if (tig == 0) {
                  const float lo = w > 0 ? sm_l[row] * a : 0.f;
                  sm_l[row] = lo + l_r[h2] * bsc;
                  sm_m[row] = Mx;
                }
              }
            }
            named_sync(2, kAttnWarps * 32);
          }
          if (ar.active) {
            for (int i = tid; i < G * (D + 2); i += kAttnWarps * 32) {
              const int row = i / (D + 2), k = i % (D + 2);
              const float v = k < D ? sm_o[row * D + k] : (k == D ? sm_m[row] : sm_l[row]);
              p.part[((size_t)(ar.g * G + row) * p.S + ar.s) * (D + 4) + k] = v;
            }
          }
        }
      } else if (ph == kPhComb) {
        // ---------------------------------------------------- combine splits
        const int P = p.Hq * D;
        const int p0 = (int)((int64_t)blockIdx.x * P / gridDim.x);
        const int p1 = (int)((int64_t)(blockIdx.x + 1) * P / gridDim.x);
        constexpr int kMaxSL = 8;  // splits per lane (S <= 256)
        for (int pi = p0 + warp; pi < p1; pi += kCW) {
          const int hq = pi / D, d = pi % D;
          const float* base = p.part + (size_t)hq * p.S * (D + 4);
          float ms[kMaxSL], ls[kMaxSL], os[kMaxSL];
#pragma unroll
          for (int k = 0; k < kMaxSL; ++k) {
            const int sp = lane + 32 * k;
            const float* ps = base + (size_t)sp * (D + 4);
            const bool in = sp < p.S;
            ms[k] = in ? __ldcg(ps + D) : -INFINITY;
            ls[k] = in ? __ldcg(ps + D + 1) : 0.f;
            os[k] = in ? __ldcg(ps + d) : 0.f;
          }
          float M = -INFINITY;
#pragma unroll
          for (int k = 0; k < kMaxSL; ++k) M = fmaxf(M, ms[k]);
          M = warp_max(M);
          float Ls = 0.f, Os = 0.f;
#pragma unroll
          for (int k = 0; k < kMaxSL; ++k) {
            const float w = (ms[k] == -INFINITY) ? 0.f : exp2f(ms[k] - M);
            Ls += ls[k] * w;
            Os += os[k] * w;
          }
          Ls = warp_sum(Ls);
          Os = warp_sum(Os);
          if (lane == 0) p.attn16[pi] = __float2half_rn(Os / Ls);
        }
      } else {
        // ---------------------------------------------------- projections
        const PhaseRows R = phase_rows(p, ph);
        if (ph == kPhQKV) {
          const PhaseRows RO = phase_rows(p, kPhO);   // rows whose residual we keep
          stage_rmsnorm16(x_l, Ly.ln1, p.H, p.eps, xs, red, RO.first, RO.first + RO.units, xres);
        } else if (ph == kPhGU) {
          stage_rmsnorm32(p.h32, Ly.ln2, p.H, p.eps, xs, red);
        } else if (ph == kPhO && p.fold) {
          stage_combine<D>(p, xs);
        } else {
          stage_copy(ph == kPhO ? p.attn16 : p.act16, R.K, xs);
        }
        // y[q] = W[q] . x on the tensor cores: A = 16 staged rows x 16
        // columns (ldmatrix), B = x as the only non-zero column, fp32
        // accumulators; the warps split each stage's 16-column steps.
        const int tg = lane & 3;
        for (int g0 = 0, gi = 0; g0 < R.nrows; g0 += kGroupRows, ++gi) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          for (int kc = 0; kc < R.ncol; ++kc) {
            int s;
            if (!take(s)) break;
            const int nks = min(kKc, R.K - kc * kKc) / 16;
            const int ks0 = warp * nks / kCW, ks1 = (warp + 1) * nks / kCW;
            const uint32_t st = smem_u32(ring + (size_t)s * kStageBytes);
            const int m = lane >> 3;
            const uint32_t arow = st + ((lane & 7) + (m & 1) * 8) * kRowStride + (m >> 1) * 16;
            const __half* xk = xs + kc * kKc + 2 * tg;
            for (int ks = ks0; ks < ks1; ++ks) {
              uint32_t a[4];
              ldsm_x4(arow + ks * 32, a);
              uint32_t b0 = 0u, b1 = 0u;
              if (lane < 4) {
                b0 = *reinterpret_cast<const uint32_t*>(xk + ks * 16);
                b1 = *reinterpret_cast<const uint32_t*>(xk + ks * 16 + 8);
              }
              mma16816(d, a, b0, b1);
            }
            give(s);
          }
          if (tg == 0) {  // column 0 of the 16 x 8 accumulator: rows lane/4 and lane/4 + 8
            float* pr = part + (gi * kCW + warp) * 16;
            pr[lane >> 2] = d[0];
            pr[(lane >> 2) + 8] = d[2];
          }
        }
        named_sync(1, kCT);
        if (*abort_flag) return;
        auto val = [&](int q) {  // fixed-order sum over the warps' partials
          const float* pr = part + (q / kGroupRows) * kCW * 16 + q % kGroupRows;
          float a = 0.f;
#pragma unroll
          for (int w = 0; w < kCW; ++w) a += pr[w * 16];
          return a;
        };
        if (ph == kPhQKV) {
          for (int k = tid; k < R.units; k += kCT) {
            const int u = R.first + k, hd = u / half, i = u % half;
            float lo = val(k), hi = val(R.units + k);
            if (hd < p.Hq) {
              if (Ly.bq) {
                lo += __half2float(Ly.bq[hd * D + i]);
                hi += __half2float(Ly.bq[hd * D + half + i]);
              }
              const float2 cs = rope_cs(p.rope, p.rope_len, half, pos, i, p.err);
              p.q32[hd * D + i] = lo * cs.x - hi * cs.y;
              p.q32[hd * D + half + i] = hi * cs.x + lo * cs.y;
            } else if (hd < p.Hq + p.Hkv) {
              const int g = hd - p.Hq;
              if (Ly.bk) {
                lo += __half2float(Ly.bk[g * D + i]);
                hi += __half2float(Ly.bk[g * D + half + i]);
              }
              const float2 cs = rope_cs(p.rope, p.rope_len, half, pos, i, p.err);
              const __half a = __float2half_rn(lo * cs.x - hi * cs.y);
              const __half bb = __float2half_rn(hi * cs.x + lo * cs.y);
              __half* dst = Ly.kc + ((size_t)g * p.max_ctx + L) * D;
              dst[i] = a;
              dst[half + i] = bb;
              if (Ly.k_new) {
                Ly.k_new[g * D + i] = a;
                Ly.k_new[g * D + half + i] = bb;
              }
            } else {
              const int g = hd - p.Hq - p.Hkv;
              if (Ly.bv) {
                lo += __half2float(Ly.bv[g * D + i]);
                hi += __half2float(Ly.bv[g * D + half + i]);
              }
              const __half a = __float2half_rn(lo), bb = __float2half_rn(hi);
              __half* dst = Ly.vc + ((size_t)g * p.max_ctx + L) * D;
              dst[i] = a;
              dst[half + i] = bb;
              if (Ly.v_new) {
                Ly.v_new[g * D + i] = a;
                Ly.v_new[g * D + half + i] = bb;
              }
            }
          }
        } else if (ph == kPhO) {
          const int r0 = R.first;
          for (int k = tid; k < R.units; k += kCT) {
            const float hv = val(k) + xres[k];
            p.h32[r0 + k] = hv;
            hres[k] = hv;   // the down phase owns the same rows
          }
        } else if (ph == kPhGU) {
          const int j0 = R.first;
          for (int k = tid; k < R.units; k += kCT)
            p.act16[j0 + k] = __float2half_rn(silu(val(k)) * val(R.units + k));
        } else {
          const int r0 = R.first;
          __half* y = layer_output(p, l);
          for (int k = tid; k < R.units; k += kCT)
            y[r0 + k] = __float2half_rn(val(k) + hres[k]);
        }
      }
      trace_point(p, l, ph, 1);
      if (l == p.n_layers - 1 && ph == kPhDown) break;  // last phase of the step
      grid_arrive(sync);
    }
  }
}

}  // namespace

// ---------------------------------------------------------------- host side

size_t decode_ws_bytes(int H, int Hq, int Hkv, int D, int I, int num_sms) {
  const size_t S = (size_t)(num_sms / Hkv);
  auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
  size_t o = 0;
  o += al((size_t)H * 2) * 2;               // xbuf0, xbuf1
  o += al((size_t)Hq * D * 4);              // q32
  o += al((size_t)Hq * S * (D + 4) * 4);    // part
  o += al((size_t)Hq * D * 2);              // attn16
  o += al((size_t)H * 4);                   // h32
  o += al((size_t)I * 2);                   // act16
  o += 256;                                 // barrier counter
  return o;
}

void decode_ws_carve(DecodeParams& p, void* ws, int num_sms) {
  const size_t S = (size_t)(num_sms / p.Hkv);
  auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
  uint8_t* b = static_cast<uint8_t*>(ws);
  size_t o = 0;
  p.xbuf0 = reinterpret_cast<__half*>(b + o); o += al((size_t)p.H * 2);
  p.xbuf1 = reinterpret_cast<__half*>(b + o); o += al((size_t)p.H * 2);
  p.q32 = reinterpret_cast<float*>(b + o); o += al((size_t)p.Hq * p.D * 4);
  p.part = reinterpret_cast<float*>(b + o); o += al((size_t)p.Hq * S * (p.D + 4) * 4);
  p.attn16 = reinterpret_cast<__half*>(b + o); o += al((size_t)p.Hq * p.D * 2);
  p.h32 = reinterpret_cast<float*>(b + o); o += al((size_t)p.H * 4);
  p.act16 = reinterpret_cast<__half*>(b + o); o += al((size_t)p.I * 2);
  p.barrier = reinterpret_cast<unsigned*>(b + o);
  // One 64-slot tile per split while there are CTAs for it (more slots per
  // split beyond that); with at most 32 splits their partials are merged in
  // the o_proj staging instead of a separate phase.
  const int64_t want = (p.cache_len + 1 + 63) / 64;
  p.S = (int)(want < 1 ? 1 : (want > (int64_t)S ? (int64_t)S : want));
  p.fold = p.S <= 32 ? 1 : 0;
}

cudaError_t launch_decode_persistent(DecodeParams& p, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.barrier, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.D == 128) return cudaLaunchKernelEx(&cfg, decode_persistent_kernel<128>, p);
  if (p.D == 64) return cudaLaunchKernelEx(&cfg, decode_persistent_kernel<64>, p);
  return cudaErrorInvalidValue;
}

cudaError_t configure_decode_persistent() {
  const cudaError_t e = cudaFuncSetAttribute(
      decode_persistent_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_persistent_kernel<64>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

}  // namespace blk
