// Decode: one token through a stack of decoder blocks in ONE persistent,
// cooperative kernel launch.
//
// At one token every projection is a matrix-vector product: the step is
// bound by the bytes of the weights (93.6 MB per 1.5B-shaped layer) and of
// the KV history.  Those bytes never depend on the token being decoded, so
// each CTA (one per SM) has a producer lane that streams, in consumption
// order, every weight box and every KV-history tile the CTA will use —
// across phase and layer boundaries — into a 4 x 48 KB shared-memory ring.
// Every copy is a TMA tensor copy with 128-byte swizzle: a weight box is 8
// rows x 1536 columns (one 3-D copy of 24 column blocks of 64), a KV tile
// 64 slots x D.  Twelve consumer warps run the phases of each layer and meet
// at a grid-wide barrier between phases.  The producer fills the ring ahead
// across phases, but issues nothing from a phase's last chunk until the next
// phase's inputs are staged: the barrier's polls and the staging loads of an
// SM wait behind every byte that SM has in flight.
//
// Phases of one layer (the block of the TopOp paper, Listing 2, at T = 1):
//   QKV   x = previous layer's output (or the input), RMSNorm(x) staged in
//         shared memory; a work unit is rows i0..i0+7 and their RoPE partners
//         i0+D/2.. of one head of wq|wk|wv; epilogue: bias, RoPE, q (fp32) to
//         the workspace, K/V to cache slot cache_len and to k_new / v_new.
//   ATTN  CTA (kv head g, split s) covers slots [j0, j1) of [0, cache_len];
//         4 warps run mma.sync m16n8k16 (rows = the G query heads of the
//         group, padded to 16) over 64-slot tiles: S = Q K^T, online softmax
//         in base 2, O += P V; the warps' states are merged and one partial
//         (acc, max, sum) per query head is written.
//   COMB  every CTA merges all splits for a slice of (head, d) pairs -> attn.
//   O     two 8-row units of wo; epilogue h = acc + x (fp32).
//   GU    RMSNorm(h) staged; unit = 8 rows of w_gate and the same 8 rows of
//         w_up; epilogue silu(gate) * up (fp16).
//   DOWN  split over (16 rows, 1536 columns) items for balance; each item's
//         fp32 partial goes to the workspace and the next reader adds the
//         partials of a row in a fixed order to h: that sum, rounded to fp16,
//         is the layer's output.
// A final phase writes the last layer's output.  Dot products are split over
// warps with fp32 accumulation; partials are added in a fixed order, so the
// result does not depend on timing.
//
// Every wait (ring mbarriers, grid barrier) is bounded; on a timeout the
// kernel records an error, stops, lets its issued copies land and returns.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "decode_persistent.h"

namespace blk {
namespace {

// 12 consumer warps + 1 producer warp: 13 warps, so no SM sub-partition holds
// more than 4 and each thread may use up to 128 registers without spilling.
constexpr int kCW = 12;                 // consumer warps
constexpr int kCT = kCW * 32;           // consumer threads
constexpr int kThreads = kCT + 32;      // + one producer warp
// Weight formats of the projections (the ABI's BLK_WFMT_* values).
enum WFmt { kF16 = 0, kI8 = 1, kU4 = 2 };
// Ring geometry per weight format.  A chunk is always 16 weight rows x kKc
// columns: 48 KB of fp16, 24 KB of INT8 codes, 12 KB of packed int4 codes.
// With fp16 weights a K/V tile (64 slots of K and V, 32 KB at D = 128) is
// one ring item; with quantized weights the stages are sized to the weight
// chunk (at least the 16 KB of one half tile), a K/V tile is two items (K,
// then V), and 16 KB stay for the phase's scales.  The ring then holds 7
// (INT8) or 11 (int4) weight chunks instead of 4.
template <int FMT> struct Ring {
  static constexpr int kStages = FMT == kF16 ? 4 : (FMT == kI8 ? 7 : 11);
  static constexpr int kStageBytes = FMT == kF16 ? 48 * 1024 : (FMT == kI8 ? 24 : 16) * 1024;
  static constexpr int kKvItems = FMT == kF16 ? 1 : 2;   // ring items per K/V tile
  static constexpr int kBoxCB = FMT == kF16 ? 24 : (FMT == kI8 ? 12 : 6);  // 128-byte blocks per box row
  static constexpr int kBoxBytes = 8 * 128 * kBoxCB;   // one 8-row box
  static constexpr int kQsBytes = FMT == kF16 ? 0 : 16 * 1024;
};
constexpr int kMaxStages = 11;
constexpr int kQsEntries = 5120;        // staged scales (and zero points) per phase
constexpr int kAttnWarps = 4;           // 4 x 16 slots = one 64-slot tile
constexpr int kSlots = 64;
constexpr int kBoxRows = 8;             // weight rows per TMA box
constexpr int kCB = 24;                 // 64-column blocks per fp16 box
constexpr int kKc = kCB * 64;           // weight columns per chunk (every format)
constexpr int kBatch = 10;              // groups whose partials shared memory holds
constexpr int kPartFloats = 2048;       // [group][warp][16] partial sums
constexpr int kQStride = 136;           // Q tile row stride in halves (padded)
static_assert(2 * Ring<kF16>::kBoxBytes <= Ring<kF16>::kStageBytes, "stage too small");
static_assert(2 * Ring<kI8>::kBoxBytes <= Ring<kI8>::kStageBytes, "stage too small");
static_assert(2 * Ring<kU4>::kBoxBytes <= Ring<kU4>::kStageBytes, "stage too small");
static_assert(64 * 128 * 2 <= Ring<kU4>::kStageBytes, "a K or V half tile fits a stage");
static_assert(kBatch * kCW * 16 <= kPartFloats, "partials too small");

constexpr int kResRows = 152;           // hidden rows per CTA (o_proj)
// shared memory layout: ring | staged input vector | partial sums (also the
// Q tile) | mbarriers and flags | o_proj residual slice | staged scales
template <int FMT> struct Smem {
  static constexpr int kXsOff = Ring<FMT>::kStages * Ring<FMT>::kStageBytes;
  static constexpr int kPartOff = kXsOff + kDecMaxVec * 2;
  static constexpr int kQOff = kPartOff;
  static constexpr int kBarOff = kPartOff + kPartFloats * 4;
  static constexpr int kResOff = kBarOff + 512;
  static constexpr int kQsOff = kResOff + kResRows * 4;
  static constexpr int kUsed = kQsOff + Ring<FMT>::kQsBytes;
  static constexpr int kBytes = kUsed + 1024;   // + alignment slack
};
static_assert(Smem<kF16>::kBytes <= 227 * 1024 && Smem<kU4>::kBytes <= 227 * 1024, "smem");

enum Phase { kPhQKV = 0, kPhAttn = 1, kPhComb = 2, kPhO = 3, kPhGU = 4, kPhDown = 5 };
// weight roles, the order of DecodeParams::tm_w
enum Role { kWq = 0, kWk = 1, kWv = 2, kWo = 3, kWg = 4, kWu = 5, kWd = 6 };
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

__device__ __forceinline__ void tma_load_2d_u32(uint32_t dst, const CUtensorMap* map, int x,
                                                int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
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

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Four INT8 codes (bytes of r, in k order) to two fp16 pairs scaled by s.
// Byte b + 128 placed under the exponent field of 1024 (fp16 0x6400) is the
// fp16 value 1024 + b + 128, exactly (the spacing of fp16 at 1024 is 1), so
// subtracting 1152 gives the code b exactly; the product with the scale is
// the one rounding.
__device__ __forceinline__ void i8x4_scaled(uint32_t r, __half2 s, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = r ^ 0x80808080u;
  const __half2 off = __float2half2_rn(1152.f);
  lo = h2_as_u32(__hmul2(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4140)), off), s));
  hi = h2_as_u32(__hmul2(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4342)), off), s));
}

// Four 4-bit codes (nibbles of v, in k order, the first in the low nibble)
// minus the zero point z, scaled by s; 1024 + c and 1024 + z are exact fp16
// values, so c - z is exact before the scaling.
__device__ __forceinline__ void u4x4_scaled(uint32_t v, uint32_t z, __half2 s, uint32_t& lo,
                                            uint32_t& hi) {
  const uint32_t a = 0x64006400u | (v & 0xFu) | ((v & 0xF0u) << 12);
  const uint32_t b = 0x64006400u | ((v >> 8) & 0xFu) | ((v & 0xF000u) << 4);
  const __half2 off = u32_as_h2((0x6400u + z) * 0x10001u);
  lo = h2_as_u32(__hmul2(__hsub2(u32_as_h2(a), off), s));
  hi = h2_as_u32(__hmul2(__hsub2(u32_as_h2(b), off), s));
}

// Address of the 16-byte chunk `ch` (8 halves) of row `r` in a 64-row tile
// stored as 128-byte-swizzled half tiles of 64 columns (8 KB each).
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int ch) {
  const int half = ch >> 3, c = ch & 7;
  return base + half * 8192 + r * 128 + ((c ^ (r & 7)) << 4);
}

// ------------------------------------------------------------ schedule
// The work of a projection phase is a list of units of 8 weight rows; a CTA
// owns a contiguous range of them, and a "group" is what one ring chunk (two
// 8-row boxes = the 16 rows of an mma tile) holds for one or more column
// chunks of 1536:
//   QKV   group = unit u: head hd, rows i0..i0+7 (tile rows 0-7) and their
//         RoPE partners i0+D/2.. (tile rows 8-15); all column chunks of H
//   O     group = two consecutive units (the second may be absent)
//   GU    group = unit u: rows 8u.. of w_gate (tile rows 0-7) and of w_up
//   DOWN  group = item (row pair p = rows 16p..16p+15, column chunk kc):
//         one column chunk each, so the 6+ chunks of a row pair spread over
//         CTAs and every CTA streams about the same number of bytes.
struct PhaseWork {
  int first, count;   // this CTA's units (DOWN: items)
  int ngroups;
  int ncol;           // column chunks of the phase's K
  int K;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

template <int D>
__device__ __forceinline__ PhaseWork phase_work(const DecodeParams& p, int ph) {
  const int b = blockIdx.x, G = gridDim.x;
  PhaseWork w;
  int total;
  if (ph == kPhQKV) { total = (p.Hq + 2 * p.Hkv) * (D / 16); w.K = p.H; }
  else if (ph == kPhO) { total = p.H / kBoxRows; w.K = p.Hq * D; }
  else if (ph == kPhGU) { total = p.I / kBoxRows; w.K = p.H; }
  else { total = ceil_div(p.H, 2 * kBoxRows) * ceil_div(p.I, kKc); w.K = p.I; }
  w.ncol = ceil_div(w.K, kKc);
  w.first = (int)((int64_t)b * total / G);
  w.count = (int)((int64_t)(b + 1) * total / G) - w.first;
  w.ngroups = ph == kPhO ? ceil_div(w.count, 2) : w.count;
  return w;
}

// What one group loads: box A (tile rows 0-7) and, unless yb < 0, box B
// (tile rows 8-15), over column chunks [ka, kb).
struct GroupDesc {
  int ra, ya, rb, yb;   // role and first row of each box
  int ka, kb;
};

template <int D>
__device__ __forceinline__ GroupDesc group_desc(const DecodeParams& p, int ph,
                                                const PhaseWork& w, int gi) {
  GroupDesc g;
  g.ka = 0;
  g.kb = w.ncol;
  if (ph == kPhQKV) {
    constexpr int upd = D / 16;  // units per head
    const int u = w.first + gi, hd = u / upd, i0 = (u % upd) * kBoxRows;
    int local;
    if (hd < p.Hq) { g.ra = kWq; local = hd; }
    else if (hd < p.Hq + p.Hkv) { g.ra = kWk; local = hd - p.Hq; }
    else { g.ra = kWv; local = hd - p.Hq - p.Hkv; }
    g.rb = g.ra;
    g.ya = local * D + i0;
    g.yb = g.ya + D / 2;
  } else if (ph == kPhO) {
    const int u = w.first + 2 * gi;
    g.ra = g.rb = kWo;
    g.ya = u * kBoxRows;
    g.yb = u + 1 < w.first + w.count ? g.ya + kBoxRows : -1;
  } else if (ph == kPhGU) {
    const int u = w.first + gi;
    g.ra = kWg; g.rb = kWu;
    g.ya = g.yb = u * kBoxRows;
  } else {
    const int it = w.first + gi, pr = it / w.ncol;
    g.ka = it % w.ncol;
    g.kb = g.ka + 1;
    g.ra = g.rb = kWd;
    g.ya = pr * 2 * kBoxRows;
    g.yb = g.ya + kBoxRows < p.H ? g.ya + kBoxRows : -1;
  }
  return g;
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
  const int64_t lo = window_lo(p.window, p.cache_len);   // slots [lo, cache_len]
  a.j0 = a.active ? lo + (int64_t)a.s * (n - lo) / p.S : 0;
  a.j1 = a.active ? lo + (int64_t)(a.s + 1) * (n - lo) / p.S : 0;
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
  // release: the CTA's writes (ordered before this by the named barrier)
  // are visible to whoever acquires the counter value that includes it
  if (threadIdx.x == 0)
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(s.counter) : "memory");
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

constexpr int kMaxNC = (kDecMaxVec + kKc - 1) / kKc;        // column chunks of DOWN

// The layer input x, four elements at float4 index i: x_in (fp16) for the
// first layer of a launch, else fp16(h + the DOWN partials of the previous
// layer, added in column-chunk order) - that layer's output.
__device__ __forceinline__ float4 layer_x4(const __half* x16, const float* h, const float* pdown,
                                           int nc, int K, int i) {
  if (x16) {
    const uint2 raw = __ldcg(reinterpret_cast<const uint2*>(x16) + i);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  float4 d[kMaxNC];
#pragma unroll
  for (int c = 0; c < kMaxNC; ++c)
    d[c] = c < nc ? __ldcg(reinterpret_cast<const float4*>(pdown + (size_t)c * K) + i)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 a = __ldcg(reinterpret_cast<const float4*>(h) + i);
#pragma unroll
  for (int c = 0; c < kMaxNC; ++c) {
    if (c < nc) { a.x += d[c].x; a.y += d[c].y; a.z += d[c].z; a.w += d[c].w; }
  }
  a.x = __half2float(__float2half_rn(a.x));
  a.y = __half2float(__float2half_rn(a.y));
  a.z = __half2float(__float2half_rn(a.z));
  a.w = __half2float(__float2half_rn(a.w));
  return a;
}

// QKV staging: xs = fp16(x * rsqrt(mean(x^2) + eps) * g) for the layer input
// x (see layer_x4); x[cap_lo, cap_hi) is also kept in cap[] for the o_proj
// residual.  x itself (fp16-exact) is parked in xs between the two passes.
__device__ void stage_qkv(const __half* x16, const float* h, const float* pdown, int nc, int K,
                          const __half* g, float eps, __half* xs, float* red, int cap_lo,
                          int cap_hi, float* cap) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nv = K / 4;
  const uint2* g2 = reinterpret_cast<const uint2*>(g);
  const uint2 g_first = tid < nv ? __ldg(g2 + tid) : make_uint2(0u, 0u);  // early
  float ss = 0.f;
#pragma unroll 1
  for (int i = tid; i < nv; i += kCT) {
    const float4 v = layer_x4(x16, h, pdown, nc, K, i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * i + e >= cap_lo && 4 * i + e < cap_hi) cap[4 * i + e - cap_lo] = f[e];
    uint2 o;
    *reinterpret_cast<__half2*>(&o.x) = __floats2half2_rn(v.x, v.y);
    *reinterpret_cast<__half2*>(&o.y) = __floats2half2_rn(v.z, v.w);
    reinterpret_cast<uint2*>(xs)[i] = o;
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  named_sync(1, kCT);
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kCW; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)K + eps);
  for (int i = tid; i < nv; i += kCT) {
    const uint2 graw = i == tid ? g_first : __ldg(g2 + i);
    const uint2 xraw = reinterpret_cast<const uint2*>(xs)[i];
    const float2 ga = __half22float2(*reinterpret_cast<const __half2*>(&graw.x));
    const float2 gb = __half22float2(*reinterpret_cast<const __half2*>(&graw.y));
    const float2 xa = __half22float2(*reinterpret_cast<const __half2*>(&xraw.x));
    const float2 xb = __half22float2(*reinterpret_cast<const __half2*>(&xraw.y));
    uint2 o;
    *reinterpret_cast<__half2*>(&o.x) = __floats2half2_rn(xa.x * r * ga.x, xa.y * r * ga.y);
    *reinterpret_cast<__half2*>(&o.y) = __floats2half2_rn(xb.x * r * gb.x, xb.y * r * gb.y);
    reinterpret_cast<uint2*>(xs)[i] = o;
  }
  named_sync(1, kCT);
}

// Same for fp32 x (the residual stream h).
__device__ void stage_rmsnorm32(const float* x, const __half* g, int K, float eps, __half* xs,
                                float* red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nv = K / 4;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const uint2* g2 = reinterpret_cast<const uint2*>(g);
  float4 v[kMaxV32];
  uint2 gr[kMaxV32];   // the gains travel with x: one round trip for both
#pragma unroll
  for (int k = 0; k < kMaxV32; ++k) {
    const int i = tid + k * kCT;
    v[k] = i < nv ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    gr[k] = i < nv ? __ldg(g2 + i) : make_uint2(0u, 0u);
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
#pragma unroll
  for (int k = 0; k < kMaxV32; ++k) {
    const int i = tid + k * kCT;
    if (i < nv) {
      const uint2 graw = gr[k];
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

// Bytes of one attention partial: acc / sum as D fp16 values, then the
// split's (max, sum) as float2, padded to 16 bytes.
__host__ __device__ constexpr int part_row_bytes(int D) { return 2 * D + 16; }

// o_proj input when the attention used few splits: xs[h*D + d] = attention
// output of query head h, merged here from the S <= 32 split partials
// instead of in a separate phase.  One warp per head: lane s loads the
// (max, sum) of split s, every lane the D/32 values it owns for every split,
// all in one round trip.
template <int D>
__device__ void stage_combine(const DecodeParams& p, __half* xs) {
  constexpr int kDL = D / 32;   // d values per lane
  constexpr int kRB = part_row_bytes(D);
  constexpr int kMaxS = 32;
  using Raw = typename std::conditional<kDL == 4, uint2, uint32_t>::type;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S;
  for (int hq = warp; hq < p.Hq; hq += kCW) {
    const uint8_t* base = p.part + (size_t)hq * S * kRB;
    const float2 ml = lane < S ? __ldcg(reinterpret_cast<const float2*>(base + (size_t)lane * kRB + 2 * D))
                               : make_float2(-INFINITY, 0.f);
    Raw a[kMaxS];
#pragma unroll
    for (int j = 0; j < kMaxS; ++j) {
      if (j < S) a[j] = __ldcg(reinterpret_cast<const Raw*>(base + (size_t)j * kRB) + lane);
      else a[j] = Raw{};
    }
    // weight of split s: exp2(m_s - M) * l_s (its values are already / l_s)
    const float M = warp_max(ml.x);
    const float wl = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M) * ml.y;
    const float Ls = warp_sum(wl);
    float o[kDL];
#pragma unroll
    for (int e = 0; e < kDL; ++e) o[e] = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxS; ++j) {
      const float w = __shfl_sync(0xffffffffu, wl, j);
      if (j < S) {
        const __half2* h = reinterpret_cast<const __half2*>(&a[j]);
#pragma unroll
        for (int e = 0; e < kDL / 2; ++e) {
          const float2 f = __half22float2(h[e]);
          o[2 * e] += f.x * w;
          o[2 * e + 1] += f.y * w;
        }
      }
    }
    const float inv = 1.f / Ls;
#pragma unroll
    for (int e = 0; e < kDL; e += 2)
      *reinterpret_cast<__half2*>(xs + hq * D + lane * kDL + e) =
          __floats2half2_rn(o[e] * inv, o[e + 1] * inv);
  }
  named_sync(1, kCT);
}

// Rows and K of weight role r.
__device__ __forceinline__ void role_shape(const DecodeParams& p, int r, int& rows, int& K) {
  const int QD = p.Hq * p.D, KD = p.Hkv * p.D;
  if (r == kWq) { rows = QD; K = p.H; }
  else if (r == kWk || r == kWv) { rows = KD; K = p.H; }
  else if (r == kWo) { rows = p.H; K = QD; }
  else if (r == kWg || r == kWu) { rows = p.I; K = p.H; }
  else { rows = p.H; K = p.I; }
}

// Quantized weights: scales staged per tile row of a work group.  INT8 has
// one scale per row; int4 one scale and one zero point per `group` columns
// of the work group's column range (all of K, or the one column chunk of a
// down-projection item).
template <int FMT>
__host__ __device__ __forceinline__ int qs_groups(int ph, int K, int group) {
  if (FMT != kU4) return 1;
  return ph == kPhDown ? (K < kKc ? K : kKc) / group : K / group;
}

// Quantized weights: a CTA's scales (and int4 zero points) of one projection
// phase, staged into shared memory as entry (gi * 16 + m) * GM + j for tile
// row m of work group gi and scale group j; rows past the matrix get scale
// 0.  qscale_load issues every load into registers before the phase's input
// staging, so both cost one round trip; qscale_store writes them after it.
constexpr int kQsPer = (kQsEntries + kCT - 1) / kCT;
struct QsRegs {
  uint16_t s[kQsPer];
  uint8_t z[kQsPer];
};

template <int D, int FMT>
__device__ __forceinline__ void qscale_load(const DecodeParams& p, int l, int ph,
                                            const PhaseWork& W, QsRegs& q) {
  const int GM = qs_groups<FMT>(ph, W.K, p.qgroup);
  const int total = W.ngroups * 16 * GM;   // <= kQsEntries, checked on the host
#pragma unroll
  for (int k = 0; k < kQsPer; ++k) {
    const int e = threadIdx.x + k * kCT;
    q.s[k] = 0;
    q.z[k] = 0;
    if (e < total) {
      const int j = e % GM, m = (e / GM) & 15, gi = e / (16 * GM);
      const GroupDesc g = group_desc<D>(p, ph, W, gi);
      const int r = m < kBoxRows ? g.ra : g.rb;
      const int y = m < kBoxRows ? g.ya + m : (g.yb >= 0 ? g.yb + m - kBoxRows : -1);
      int rows, K;
      role_shape(p, r, rows, K);
      if (y >= 0 && y < rows) {
        if (FMT == kI8) {
          q.s[k] = __ldg(p.qscale[l][r] + y);
        } else {
          const int ng = K / p.qgroup, jg = g.ka * kKc / p.qgroup + j;
          if (jg < ng) {
            q.s[k] = __ldg(p.qscale[l][r] + (size_t)y * ng + jg);
            q.z[k] = __ldg(p.qzero[l][r] + (size_t)y * ng + jg);
          }
        }
      }
    }
  }
}

template <int FMT>
__device__ __forceinline__ void qscale_store(const DecodeParams& p, int ph, const PhaseWork& W,
                                             const QsRegs& q, __half* qs_s, uint8_t* qs_z) {
  const int total = W.ngroups * 16 * qs_groups<FMT>(ph, W.K, p.qgroup);
#pragma unroll
  for (int k = 0; k < kQsPer; ++k) {
    const int e = threadIdx.x + k * kCT;
    if (e < total) {
      qs_s[e] = __ushort_as_half(q.s[k]);
      if (FMT == kU4) qs_z[e] = q.z[k];
    }
  }
  named_sync(1, kCT);
}

// Position in this CTA's stream of ring chunks: layer l, phase ph, and
// within the phase either the K/V tile c or (group gi, column chunk kc).
struct Cursor {
  int l, ph, c, gi, kc;
  PhaseWork W;
  GroupDesc g;
};

// Settles on the first chunk at or after (l, ph); false past the last layer.
template <int D>
__device__ bool cursor_begin(Cursor& cu, const DecodeParams& p, const AttnRange& ar,
                             int kv_items) {
  for (; cu.l < p.n_layers; ++cu.l, cu.ph = 0) {
    for (; cu.ph < kPhases; ++cu.ph) {
      if (cu.ph == kPhComb) continue;
      if (cu.ph == kPhAttn) {
        if (ar.chunks > 0) { cu.c = 0; return true; }
        continue;
      }
      cu.W = phase_work<D>(p, cu.ph);
      if (cu.W.ngroups > 0) {
        cu.gi = 0;
        cu.g = group_desc<D>(p, cu.ph, cu.W, 0);
        cu.kc = cu.g.ka;
        return true;
      }
    }
  }
  return false;
}

template <int D>
__device__ bool cursor_next(Cursor& cu, const DecodeParams& p, const AttnRange& ar,
                            int kv_items) {
  if (cu.ph == kPhAttn) {
    if (++cu.c < ar.chunks * kv_items) return true;
  } else {
    if (++cu.kc < cu.g.kb) return true;
    if (++cu.gi < cu.W.ngroups) {
      cu.g = group_desc<D>(p, cu.ph, cu.W, cu.gi);
      cu.kc = cu.g.ka;
      return true;
    }
  }
  ++cu.ph;
  return cursor_begin<D>(cu, p, ar, kv_items);
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
template <int D, int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_persistent_kernel(const __grid_constant__ DecodeParams p) {
  using RG = Ring<FMT>;
  using SM = Smem<FMT>;
  constexpr int kStages = RG::kStages;
  constexpr int kStageBytes = RG::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  __half* xs = reinterpret_cast<__half*>(smem + SM::kXsOff);
  float* part = reinterpret_cast<float*>(smem + SM::kPartOff);
  __half* qtile = reinterpret_cast<__half*>(smem + SM::kQOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBarOff);
  uint64_t* empty = full + kMaxStages;
  float* red = reinterpret_cast<float*>(empty + kMaxStages);     // [16]
  // staged scales of a quantized phase: kQsEntries fp16 scales, then as many
  // int4 zero points
  __half* qs_s = reinterpret_cast<__half*>(smem + SM::kQsOff);
  uint8_t* qs_z = reinterpret_cast<uint8_t*>(qs_s + kQsEntries);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 16);
  // quiet: set from the moment the consumers take the last ring chunk of a
  // phase until they have staged the next phase's inputs.  The producer
  // issues no new copy meanwhile: the grid barrier's polls and the staging
  // loads of an SM queue behind the bytes that SM has requested, so copies
  // issued then would delay them (measured: a grid barrier took ~2.5 us with
  // copies in flight, ~1.4 us without).
  volatile int* quiet = abort_flag + 1;
  float* xres = reinterpret_cast<float*>(smem + SM::kResOff);   // x of the o_proj rows

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    *abort_flag = 0;
    *quiet = 0;
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
    // column blocks one box copy covers in chunk kc of role r
    auto box_cbs = [&](int r, int kc) -> int {
      return p.w3d[r] ? p.wbox_z[r] : min(RG::kBoxCB, p.wnz[r] - kc * RG::kBoxCB);
    };
    auto chunk_bytes = [&](const Cursor& cu) -> uint32_t {
      if (cu.ph == kPhAttn) return (uint32_t)(2 / RG::kKvItems) * kv_tile_bytes;
      const uint32_t nb = cu.g.yb >= 0 ? 2u : 1u;
      return nb * (uint32_t)(kBoxRows * 128) * (uint32_t)box_cbs(cu.g.ra, cu.kc);
    };
    auto kv_row = [&](const Cursor& cu) {
      return (int)(ar.g * p.max_ctx + ar.j0 + (int64_t)(cu.c / RG::kKvItems) * kSlots);
    };
    // one 8-row box of role r at row y, column chunk kc: a single 3-D copy,
    // or (a row not a multiple of 128 bytes) one 2-D copy per 128-byte block
    // (64 fp16 columns, 128 INT8 columns or 128 bytes of packed int4)
    auto copy_box = [&](int l, int r, int y, int kc, uint32_t dst, uint32_t bar) {
      const CUtensorMap* m = &p.tm_w[l][r];
      if (p.w3d[r]) {
        tma_load_3d(dst, m, 0, y, kc * RG::kBoxCB, bar);
      } else {
        const int n = min(RG::kBoxCB, p.wnz[r] - kc * RG::kBoxCB);
        const int epb = FMT == kF16 ? 64 : 128;   // tensor elements per block
        for (int cb = 0; cb < n; ++cb)
          tma_load_2d_u32(dst + cb * (kBoxRows * 128), m, (kc * RG::kBoxCB + cb) * epb, y, bar);
      }
    };
    auto load = [&](const Cursor& cu, uint8_t* st, uint64_t* bar) {
      if (cu.ph == kPhAttn) {
        const int y = kv_row(cu);
        if (RG::kKvItems == 1) {
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_2d(st + h * 8192, &p.tm_k[cu.l], h * 64, y, bar);
            tma_load_2d(st + kv_tile_bytes + h * 8192, &p.tm_v[cu.l], h * 64, y, bar);
          }
        } else {
          const CUtensorMap* m = (cu.c & 1) ? &p.tm_v[cu.l] : &p.tm_k[cu.l];
#pragma unroll
          for (int h = 0; h < D / 64; ++h) tma_load_2d(st + h * 8192, m, h * 64, y, bar);
        }
        return;
      }
      const uint32_t dst = smem_u32(st), mb = smem_u32(bar);
      copy_box(cu.l, cu.g.ra, cu.g.ya, cu.kc, dst, mb);
      if (cu.g.yb >= 0) copy_box(cu.l, cu.g.rb, cu.g.yb, cu.kc, dst + RG::kBoxBytes, mb);
    };
    Cursor rc = {0, 0, 0, 0, 0, {}, {}};
    bool more = cursor_begin<D>(rc, p, ar, RG::kKvItems);
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
      if (*quiet) {
        const uint64_t t0 = global_ns();
        while (*quiet && !*abort_flag) {
          if (global_ns() - t0 > kWaitLimitNs) {
            set_error(p.err, kDevTimeout);
            *abort_flag = 1;
            break;
          }
        }
        if (*abort_flag) break;
      }
      mbar_arrive_expect_tx(&full[s], chunk_bytes(rc));
      load(rc, ring + (size_t)s * kStageBytes, &full[s]);
      ++it;
      more = cursor_next<D>(rc, p, ar, RG::kKvItems);
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
  auto take = [&](int& s, int ahead = 0) -> bool {   // wait for ring item it + ahead
    const int k = it + ahead;
    s = k % kStages;
    if (*abort_flag) return false;
    if (!mbar_wait(&full[s], (k / kStages) & 1, p.err)) {
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
          if (tid == 0) *quiet = 0;
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
          int s, sv = 0;   // the stages of the tile's K and V (one stage for fp16 weights)
          if (!take(s)) break;
          if (RG::kKvItems == 2 && !take(sv, 1)) break;
          if (c == ar.chunks - 1 && tid == 0) *quiet = 1;
          if (warp < kAttnWarps) {
            uint8_t* st = ring + (size_t)s * kStageBytes;
            uint8_t* vst = RG::kKvItems == 1 ? st + kv_tile_bytes : ring + (size_t)sv * kStageBytes;
            const uint32_t kb = smem_u32(st), vb = smem_u32(vst);
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
                  *reinterpret_cast<uint4*>(vst + (tile_addr(vb, r, ch) - vb)) = kv_v;
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
          if (RG::kKvItems == 2) give(sv);
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
          // pairwise merge through two buffers {m[16], l[16], o[16][D + 8]} in
          // the staging area: warps 1, 3 -> 0, 2, then 2 -> 0.  Rows of o are
          // padded so that the float2 accesses of a warp hit distinct banks.
          constexpr int kOS = D + 8, kBuf = 32 + 16 * kOS;
          float* bufs = reinterpret_cast<float*>(xs);
          auto put = [&](float* bf) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int row = grp + 8 * h2;
              if (tig == 0) { bf[row] = m_r[h2]; bf[16 + row] = l_r[h2]; }
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
              const float bsc = (Mx == -INFINITY) ? 0.f : exp2f(m_r[h2] - Mx);
#pragma unroll
              for (int dn = 0; dn < D / 8; ++dn) {
                const float2 o = *reinterpret_cast<const float2*>(bf + 32 + row * kOS + dn * 8 + 2 * tig);
                O[dn][2 * h2] = O[dn][2 * h2] * bsc + o.x * a;
                O[dn][2 * h2 + 1] = O[dn][2 * h2 + 1] * bsc + o.y * a;
              }
              l_r[h2] = l_r[h2] * bsc + lo * a;
              m_r[h2] = Mx;
            }
          };
          if (warp & 1) put(bufs + (warp >> 1) * kBuf);
          named_sync(2, kAttnWarps * 32);
          if (!(warp & 1)) merge_from(bufs + (warp >> 1) * kBuf);
          if (warp == 2) { __syncwarp(); put(bufs + kBuf); }
          named_sync(2, kAttnWarps * 32);
          if (warp == 0) { merge_from(bufs + kBuf); put(bufs); }
          named_sync(2, kAttnWarps * 32);
          if (ar.active) {
            constexpr int kRB = part_row_bytes(D), kPairs = D / 2 + 1;
            for (int i = tid; i < G * kPairs; i += kAttnWarps * 32) {
              const int row = i / kPairs, k = i % kPairs;
              uint8_t* dst = p.part + ((size_t)(ar.g * G + row) * p.S + ar.s) * kRB;
              const float l = bufs[16 + row];
              if (k < D / 2) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const float* o = bufs + 32 + row * kOS + 2 * k;
                *reinterpret_cast<__half2*>(dst + 4 * k) = __floats2half2_rn(o[0] * inv, o[1] * inv);
              } else {
                *reinterpret_cast<float2*>(dst + 2 * D) = make_float2(bufs[row], l);
              }
            }
          }
        }
      } else if (ph == kPhComb) {
        // ---------------------------------------------------- combine splits
        if (tid == 0) *quiet = 0;
        const int P = p.Hq * D;
        const int p0 = (int)((int64_t)blockIdx.x * P / gridDim.x);
        const int p1 = (int)((int64_t)(blockIdx.x + 1) * P / gridDim.x);
        constexpr int kMaxSL = 8;  // splits per lane (S <= 256)
        for (int pi = p0 + warp; pi < p1; pi += kCW) {
          const int hq = pi / D, d = pi % D;
          constexpr int kRB = part_row_bytes(D);
          const uint8_t* base = p.part + (size_t)hq * p.S * kRB;
          float ms[kMaxSL], ls[kMaxSL], os[kMaxSL];
#pragma unroll
          for (int k = 0; k < kMaxSL; ++k) {
            const int sp = lane + 32 * k;
            const uint8_t* ps = base + (size_t)sp * kRB;
            const bool in = sp < p.S;
            const float2 ml = in ? __ldcg(reinterpret_cast<const float2*>(ps + 2 * D))
                                 : make_float2(-INFINITY, 0.f);
            ms[k] = ml.x;
            ls[k] = ml.y;
            os[k] = in ? __half2float(__ldcg(reinterpret_cast<const __half*>(ps) + d)) : 0.f;
          }
          float M = -INFINITY;
#pragma unroll
          for (int k = 0; k < kMaxSL; ++k) M = fmaxf(M, ms[k]);
          M = warp_max(M);
          float Ls = 0.f, Os = 0.f;
#pragma unroll
          for (int k = 0; k < kMaxSL; ++k) {
            const float w = (ms[k] == -INFINITY) ? 0.f : exp2f(ms[k] - M) * ls[k];
            Ls += w;
            Os += os[k] * w;
          }
          Ls = warp_sum(Ls);
          Os = warp_sum(Os);
          if (lane == 0) p.attn16[pi] = __float2half_rn(Os / Ls);
        }
      } else {
        // ---------------------------------------------------- projections
        const PhaseWork W = phase_work<D>(p, ph);
        // bias and RoPE factors of a QKV epilogue item (group gi, tile row m < 8)
        struct QkvConst { float blo, bhi; float2 cs; };
        auto qkv_const = [&](int gi, int m) {
          constexpr int upd = D / 16;
          const int u = W.first + gi, hd = u / upd, i = (u % upd) * kBoxRows + m;
          QkvConst c{0.f, 0.f, make_float2(1.f, 0.f)};
          const __half* bias;
          int row;
          if (hd < p.Hq) { bias = Ly.bq; row = hd * D; }
          else if (hd < p.Hq + p.Hkv) { bias = Ly.bk; row = (hd - p.Hq) * D; }
          else { bias = Ly.bv; row = (hd - p.Hq - p.Hkv) * D; }
          if (bias) {
            c.blo = __half2float(bias[row + i]);
            c.bhi = __half2float(bias[row + half + i]);
          }
          if (hd < p.Hq + p.Hkv) c.cs = rope_cs(p.rope, p.rope_len, half, pos, i, p.err);
          return c;
        };
        // those of this thread's item in the first batch, fetched before the
        // staging so that their latency overlaps it
        QkvConst qc0{0.f, 0.f, make_float2(1.f, 0.f)};
        if (ph == kPhQKV && tid < min(W.ngroups, kBatch) * 16 && (tid & 15) < kBoxRows)
          qc0 = qkv_const(tid >> 4, tid & 15);
        QsRegs qsr;
        if constexpr (FMT != kF16) qscale_load<D, FMT>(p, l, ph, W, qsr);
        if (ph == kPhQKV) {
          const PhaseWork WO = phase_work<D>(p, kPhO);   // rows whose residual we keep
          stage_qkv(l == 0 ? p.x_in : nullptr, p.h32, p.pdown, p.nc_down, p.H, Ly.ln1, p.eps,
                    xs, red, WO.first * kBoxRows, (WO.first + WO.count) * kBoxRows, xres);
        } else if (ph == kPhGU) {
          stage_rmsnorm32(p.h32, Ly.ln2, p.H, p.eps, xs, red);
        } else if (ph == kPhO && p.fold) {
          stage_combine<D>(p, xs);
        } else {
          stage_copy(ph == kPhO ? p.attn16 : p.act16, W.K, xs);
        }
        if constexpr (FMT != kF16) qscale_store<FMT>(p, ph, W, qsr, qs_s, qs_z);
        if (tid == 0) *quiet = 0;
        // y = W x on the tensor cores: A = a chunk's 16 rows x 16 columns
        // (ldmatrix from the two swizzled boxes), B = x as the only non-zero
        // column, fp32 accumulators; the warps split each chunk's 16-column
        // steps.  Partials of up to kBatch groups stay in shared memory and
        // the epilogue adds them in warp order.
        const int tg = lane & 3, m8 = lane >> 3, r8 = lane & 7, g8 = lane >> 2;
        const uint32_t abox = (uint32_t)((m8 & 1) * RG::kBoxBytes + r8 * 128);
        const int khalf = m8 >> 1;
        const int GM = qs_groups<FMT>(ph, W.K, p.qgroup);
        for (int b0 = 0; b0 < W.ngroups; b0 += kBatch) {
          const int b1 = min(W.ngroups, b0 + kBatch);
          for (int gi = b0; gi < b1; ++gi) {
            const GroupDesc g = group_desc<D>(p, ph, W, gi);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            for (int kc = g.ka; kc < g.kb; ++kc) {
              int s;
              if (!take(s)) break;
              if (gi == W.ngroups - 1 && kc == g.kb - 1 && tid == 0) *quiet = 1;
              const int nks = min(kKc, W.K - kc * kKc) / 16;
              const int ks0 = warp * nks / kCW, ks1 = (warp + 1) * nks / kCW;
              if constexpr (FMT == kF16) {
                const uint32_t st = smem_u32(ring + (size_t)s * kStageBytes) + abox;
                const __half* xk = xs + kc * kKc + 2 * tg;
                for (int ks = ks0; ks < ks1; ++ks) {
                  uint32_t a[4];
                  ldsm_x4(st + (ks >> 2) * 1024 + (((((ks & 3) << 1) | khalf) ^ r8) << 4), a);
                  uint32_t x0 = 0u, x1 = 0u;
                  if (lane < 4) {
                    x0 = *reinterpret_cast<const uint32_t*>(xk + ks * 16);
                    x1 = *reinterpret_cast<const uint32_t*>(xk + ks * 16 + 8);
                  }
                  mma16816(d, a, x0, x1);
                }
              } else {
                // Quantized codes: each lane reads the 4 consecutive codes
                // k = 16 ks + 4 tg .. + 3 of rows g8 (box A) and g8 + 8 (box
                // B) and makes them the A-fragment slots (2 tg, 2 tg + 1) and
                // (2 tg + 8, 2 tg + 9); x is read in the same k order, so the
                // product sums every k once.
                const uint32_t sta = smem_u32(ring + (size_t)s * kStageBytes) + g8 * 128;
                const uint32_t stb = sta + RG::kBoxBytes;
                const __half* srow = qs_s + (gi * 16 + g8) * GM;
                const uint8_t* zrow = qs_z + (gi * 16 + g8) * GM;
                const int kbase = (kc - g.ka) * kKc;
                // the scales (and zero points) change every `group` columns
                int jc = -1;
                __half2 sA = __half2half2(srow[0]), sB = __half2half2(srow[8 * GM]);
                uint32_t zA = 0, zB = 0;
                for (int ks = ks0; ks < ks1; ++ks) {
                  uint32_t a[4];
                  if constexpr (FMT == kI8) {
                    const uint32_t off = (ks >> 3) * 1024 + (((ks & 7) ^ g8) << 4) + 4 * tg;
                    i8x4_scaled(lds_u32(sta + off), sA, a[0], a[2]);
                    i8x4_scaled(lds_u32(stb + off), sB, a[1], a[3]);
                  } else {
                    const int j = (kbase + 16 * ks) >> p.qgroup_lg;
                    if (j != jc) {
                      jc = j;
                      sA = __half2half2(srow[j]);
                      sB = __half2half2(srow[8 * GM + j]);
                      zA = zrow[j];
                      zB = zrow[8 * GM + j];
                    }
                    const uint32_t off =
                        (ks >> 4) * 1024 + ((((ks & 15) >> 1) ^ g8) << 4) + 8 * (ks & 1) + 2 * tg;
                    u4x4_scaled(lds_u16(sta + off), zA, sA, a[0], a[2]);
                    u4x4_scaled(lds_u16(stb + off), zB, sB, a[1], a[3]);
                  }
                  uint32_t x0 = 0u, x1 = 0u;
                  if (lane < 4) {
                    const uint2 xv =
                        *reinterpret_cast<const uint2*>(xs + kc * kKc + 16 * ks + 4 * lane);
                    x0 = xv.x;
                    x1 = xv.y;
                  }
                  mma16816(d, a, x0, x1);
                }
              }
              give(s);
            }
            if (tg == 0) {  // column 0 of the 16 x 8 accumulator: rows lane/4 and lane/4 + 8
              float* pr = part + ((gi - b0) * kCW + warp) * 16;
              pr[lane >> 2] = d[0];
              pr[(lane >> 2) + 8] = d[2];
            }
          }
          named_sync(1, kCT);
          if (*abort_flag) return;
          auto val = [&](int gl, int m) {  // fixed-order sum over the warps' partials
            const float* pr = part + gl * kCW * 16 + m;
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) a += pr[w * 16];
            return a;
          };
          for (int e = tid; e < (b1 - b0) * 16; e += kCT) {
            const int gl = e >> 4, m = e & 15, gi = b0 + gl;
            if (ph == kPhQKV) {
              if (m >= kBoxRows) continue;
              constexpr int upd = D / 16;
              const int u = W.first + gi, hd = u / upd, i = (u % upd) * kBoxRows + m;
              const QkvConst c = b0 == 0 ? qc0 : qkv_const(gi, m);
              const float lo = val(gl, m) + c.blo, hi = val(gl, m + kBoxRows) + c.bhi;
              const float2 cs = c.cs;
              if (hd < p.Hq) {
                p.q32[hd * D + i] = lo * cs.x - hi * cs.y;
                p.q32[hd * D + half + i] = hi * cs.x + lo * cs.y;
              } else if (hd < p.Hq + p.Hkv) {
                const int gk = hd - p.Hq;
                const __half a = __float2half_rn(lo * cs.x - hi * cs.y);
                const __half bb = __float2half_rn(hi * cs.x + lo * cs.y);
                __half* dst = Ly.kc + ((size_t)gk * p.max_ctx + L) * D;
                dst[i] = a;
                dst[half + i] = bb;
                if (Ly.k_new) {
                  Ly.k_new[gk * D + i] = a;
                  Ly.k_new[gk * D + half + i] = bb;
                }
              } else {
                const int gv = hd - p.Hq - p.Hkv;
                const __half a = __float2half_rn(lo), bb = __float2half_rn(hi);
                __half* dst = Ly.vc + ((size_t)gv * p.max_ctx + L) * D;
                dst[i] = a;
                dst[half + i] = bb;
                if (Ly.v_new) {
                  Ly.v_new[gv * D + i] = a;
                  Ly.v_new[gv * D + half + i] = bb;
                }
              }
            } else if (ph == kPhO) {
              const int row = (W.first + 2 * gi) * kBoxRows + m;
              if (row < (W.first + W.count) * kBoxRows)
                p.h32[row] = val(gl, m) + xres[row - W.first * kBoxRows];
            } else if (ph == kPhGU) {
              if (m >= kBoxRows) continue;
              const int j = (W.first + gi) * kBoxRows + m;
              p.act16[j] = __float2half_rn(silu(val(gl, m)) * val(gl, m + kBoxRows));
            } else {
              const int it = W.first + gi, row = (it / W.ncol) * 2 * kBoxRows + m;
              if (row < p.H) p.pdown[(size_t)(it % W.ncol) * p.H + row] = val(gl, m);
            }
          }
          named_sync(1, kCT);   // the partials are reused by the next batch
        }
      }
      trace_point(p, l, ph, 1);
      if (tid == 0) *quiet = 1;
      grid_arrive(sync);
    }
  }
  // final phase: the last layer's output, fp16(h + its DOWN partials)
  if (!grid_wait(sync, bar++)) return;
  {
    const int nv = p.H / 4, G = gridDim.x;
    const int i0 = (int)((int64_t)blockIdx.x * nv / G), i1 = (int)((int64_t)(blockIdx.x + 1) * nv / G);
    for (int i = i0 + tid; i < i1; i += kCT) {
      const float4 v = layer_x4(nullptr, p.h32, p.pdown, p.nc_down, p.H, i);
      uint2 o;
      *reinterpret_cast<__half2*>(&o.x) = __floats2half2_rn(v.x, v.y);
      *reinterpret_cast<__half2*>(&o.y) = __floats2half2_rn(v.z, v.w);
      reinterpret_cast<uint2*>(p.out)[i] = o;
    }
  }
}

}  // namespace

// ---------------------------------------------------------------- host side

size_t decode_ws_bytes(int H, int Hq, int Hkv, int D, int I, int num_sms) {
  const size_t S = (size_t)(num_sms / Hkv);
  auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
  size_t o = 0;
  o += al((size_t)H * 4 * ((I + kKc - 1) / kKc));   // pdown
  o += al((size_t)Hq * D * 4);              // q32
  o += al((size_t)Hq * S * part_row_bytes(D));   // part
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
  p.nc_down = (p.I + kKc - 1) / kKc;
  p.pdown = reinterpret_cast<float*>(b + o); o += al((size_t)p.H * 4 * p.nc_down);
  p.q32 = reinterpret_cast<float*>(b + o); o += al((size_t)p.Hq * p.D * 4);
  p.part = b + o; o += al((size_t)p.Hq * S * part_row_bytes(p.D));
  p.attn16 = reinterpret_cast<__half*>(b + o); o += al((size_t)p.Hq * p.D * 2);
  p.h32 = reinterpret_cast<float*>(b + o); o += al((size_t)p.H * 4);
  p.act16 = reinterpret_cast<__half*>(b + o); o += al((size_t)p.I * 2);
  p.barrier = reinterpret_cast<unsigned*>(b + o);
  // One 64-slot tile per split while there are CTAs for it (more slots per
  // split beyond that); with at most 32 splits their partials are merged in
  // the o_proj staging instead of a separate phase.
  const int64_t want = (p.cache_len + 1 - window_lo(p.window, p.cache_len) + 63) / 64;
  p.S = (int)(want < 1 ? 1 : (want > (int64_t)S ? (int64_t)S : want));
  p.fold = p.S <= 32 ? 1 : 0;
}

template <int D, int FMT>
static cudaError_t launch_one(const cudaLaunchConfig_t& base, const DecodeParams& p) {
  cudaLaunchConfig_t cfg = base;
  cfg.dynamicSmemBytes = Smem<FMT>::kBytes;
  return cudaLaunchKernelEx(&cfg, decode_persistent_kernel<D, FMT>, p);
}

cudaError_t launch_decode_persistent(DecodeParams& p, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.barrier, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.D == 128) {
    if (p.fmt == kF16) return launch_one<128, kF16>(cfg, p);
    if (p.fmt == kI8) return launch_one<128, kI8>(cfg, p);
    if (p.fmt == kU4) return launch_one<128, kU4>(cfg, p);
  } else if (p.D == 64) {
    if (p.fmt == kF16) return launch_one<64, kF16>(cfg, p);
    if (p.fmt == kI8) return launch_one<64, kI8>(cfg, p);
    if (p.fmt == kU4) return launch_one<64, kU4>(cfg, p);
  }
  return cudaErrorInvalidValue;
}

template <int D, int FMT>
static cudaError_t configure_one() {
  return cudaFuncSetAttribute(decode_persistent_kernel<D, FMT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<FMT>::kBytes);
}

cudaError_t configure_decode_persistent() {
  const cudaError_t es[6] = {configure_one<128, kF16>(), configure_one<128, kI8>(),
                             configure_one<128, kU4>(),  configure_one<64, kF16>(),
                             configure_one<64, kI8>(),   configure_one<64, kU4>()};
  for (cudaError_t e : es)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

int decode_q_max_entries(int H, int Hq, int Hkv, int D, int I, int fmt, int group, int num_sms) {
  if (fmt == kF16) return 0;
  const int QD = Hq * D;
  auto per_cta = [&](int units) { return (units + num_sms - 1) / num_sms; };
  // work groups per CTA and K of each phase (see phase_work)
  const int g_qkv = per_cta((Hq + 2 * Hkv) * (D / 16));
  const int g_o = (per_cta(H / kBoxRows) + 1) / 2;
  const int g_gu = per_cta(I / kBoxRows);
  const int g_dn = per_cta(((H + 2 * kBoxRows - 1) / (2 * kBoxRows)) * ((I + kKc - 1) / kKc));
  auto gm = [&](int ph, int K) {
    return fmt == kI8 ? qs_groups<kI8>(ph, K, group) : qs_groups<kU4>(ph, K, group);
  };
  int m = g_qkv * 16 * gm(kPhQKV, H);
  m = std::max(m, g_o * 16 * gm(kPhO, QD));
  m = std::max(m, g_gu * 16 * gm(kPhGU, H));
  m = std::max(m, g_dn * 16 * gm(kPhDown, I));
  return m;
}

int decode_q_entry_limit() { return kQsEntries; }

}  // namespace blk
