// C ABI of the decoder-block library: argument validation, workspace layout
// and the kernel sequence of each phase.  See include/blk.h for the contract.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/blk.h"
#include "common.cuh"
#include "blk_internal.h"
#include "decode_persistent.h"
#include "gemm_fr.h"
#include "gemm_tc.h"
#include "kernels.h"

using namespace blk;

namespace {
constexpr int kMaxPending = 1024;
// Kernel ids for per-kernel timing (blk_timing_read).
enum KernelId {
  kKRmsNorm = 0, kKGemmQKV, kKSplitReduce, kKAttnPrefill, kKGemmO, kKGemmGateUp,
  kKGemmDown, kKDecodeStep, kKAttnMerge, kKLmHead, kKArgmax, kKEmbed, kKDecodeAttnBatch,
  kKQkvFinish, kKDequant, kKReduceNorm, kKCount
};
static_assert(kKCount <= BLK_N_KERNELS, "kernel id table");
const char* const kKernelNames[BLK_N_KERNELS] = {
    "rmsnorm_rows", "gemm_qkv", "splitk_reduce", "attn_prefill", "gemm_o",
    "gemm_gateup", "gemm_down", "decode_persistent", "attn_merge", "lm_head", "argmax_reduce",
    "embed", "decode_attn_batch", "qkv_finish", "dequant_weights", "splitk_reduce_norm"};
}  // namespace

struct blk_handle_s {
  blk_config cfg;
  int device;
  int num_sms;
  float2* rope;   // [max_ctx][head_dim / 2] (cos, sin)
  int* status;    // device status word
  uint32_t flags;
  bool decode_ok;  // shape fits the persistent decode kernel
  int64_t window;  // sliding-window attention in slots (0 = full), blk_set_window
  blk::DecodeParams* dec;  // parameter block of the decode launch
  uint64_t* trace;         // optional decode timeline buffer
  size_t trace_len;
  // per-kernel timing
  bool timing;
  bool overflow;
  cudaEvent_t* ev;  // 2 * kMaxPending, created on first blk_timing(h, 1)
  int pending;
  int pending_kernel[kMaxPending];
  double total_ms[BLK_N_KERNELS];
  int64_t launches[BLK_N_KERNELS];
};

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

bool group_supported(int g) {
  return g == 1 || g == 2 || g == 4 || g == 6 || g == 8 || g == 16;
}

int shape_ok(const blk_config* c) {
  if (c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
      c->intermediate <= 0 || c->max_ctx < 1)
    return BLK_ERR_SHAPE;
  if (c->head_dim != 64 && c->head_dim != 128) return BLK_ERR_SHAPE;
  if (c->n_heads % c->n_kv_heads != 0) return BLK_ERR_SHAPE;
  if (!group_supported(c->n_heads / c->n_kv_heads)) return BLK_ERR_SHAPE;
  if (c->hidden % 64 || c->intermediate % 8) return BLK_ERR_SHAPE;
  if ((c->n_heads * c->head_dim) % 64) return BLK_ERR_SHAPE;
  if (c->hidden > 16384 || c->intermediate > 16384) return BLK_ERR_SHAPE;
  if (c->n_heads * c->head_dim > 16384) return BLK_ERR_SHAPE;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return BLK_ERR_SHAPE;
  if (c->max_ctx > (int64_t)1 << 31) return BLK_ERR_SHAPE;
  return BLK_OK;
}

// Workspace layout.  Prefill and decode buffers start at offset 0 (a call
// uses one of the two layouts).
constexpr int kMaxSplits = 4;        // split-K partial buffers of the down projection
// Batched decode (at most a few hundred rows): QKV, o_proj and down have few
// N tiles and need K splits to occupy every SM pair.
constexpr int kMaxSplitsBatch = 16;
constexpr int kMaxSplitsNorm = 8;    // partials the split-K RMSNorm adds

struct PrefillWs {
  size_t xn16, q16, attn16, h32, hn16, act16, part32, total;
};

// part32 holds the attention's chunk partials first and the down
// projection's split-K partials later (never live at the same time).
PrefillWs prefill_ws(const blk_config& c, int64_t T, int num_sms) {
  const size_t H = c.hidden, D = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads,
               I = c.intermediate;
  (void)Hkv;
  PrefillWs w;
  size_t o = 0;
  w.xn16 = o; o = align_up(o + T * H * 2);
  w.q16 = o; o = align_up(o + T * Hq * D * 2);
  w.attn16 = o; o = align_up(o + T * Hq * D * 2);
  w.h32 = o; o = align_up(o + T * H * 4);
  w.hn16 = o; o = align_up(o + T * H * 2);
  w.act16 = o; o = align_up(o + T * I * 2);
  const size_t split_k = (size_t)kMaxSplits * T * H * 4;
  const size_t attn = prefill_attn_part_bytes(T, (int)Hq, (int)D, num_sms);
  w.part32 = o; o = align_up(o + (split_k > attn ? split_k : attn));
  w.total = o;
  return w;
}


int check_weights(const blk_config& c, const blk_weights* w) {
  if (!w) return BLK_ERR_NULL;
  const void* mats[] = {w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up, w->w_down};
  for (const void* m : mats) {
    if (!m) return BLK_ERR_NULL;
    if (!aligned(m, 16)) return BLK_ERR_ALIGN;
  }
  // gains and biases are read as 16-byte vectors, like every other operand
  if (!w->ln1_g || !w->ln2_g) return BLK_ERR_NULL;
  if (!aligned(w->ln1_g, 16) || !aligned(w->ln2_g, 16)) return BLK_ERR_ALIGN;
  if (c.has_qkv_bias) {
    if (!w->bq || !w->bk || !w->bv) return BLK_ERR_NULL;
    if (!aligned(w->bq, 16) || !aligned(w->bk, 16) || !aligned(w->bv, 16))
      return BLK_ERR_ALIGN;
  }
  return BLK_OK;
}

// Quantized weights: pointers, alignment and the shape rules of blk.h.
int check_qweights(const blk_config& c, const blk_qweights* w) {
  if (!w) return BLK_ERR_NULL;
  if (w->format != BLK_WFMT_I8 && w->format != BLK_WFMT_U4) return BLK_ERR_SHAPE;
  const int64_t Ks[3] = {c.hidden, (int64_t)c.n_heads * c.head_dim, c.intermediate};
  for (int64_t K : Ks) {
    if (K % (w->format == BLK_WFMT_I8 ? 16 : 32)) return BLK_ERR_SHAPE;
    if (w->format == BLK_WFMT_U4 &&
        (w->group < 16 || (w->group & (w->group - 1)) || K % w->group))
      return BLK_ERR_SHAPE;
  }
  const blk_qmatrix* m[] = {&w->wq, &w->wk, &w->wv, &w->wo, &w->w_gate, &w->w_up, &w->w_down};
  for (const blk_qmatrix* q : m) {
    if (!q->q || !q->scale || (w->format == BLK_WFMT_U4 && !q->zero)) return BLK_ERR_NULL;
    if (!aligned(q->q, 16) || !aligned(q->scale, 2)) return BLK_ERR_ALIGN;
  }
  if (!w->ln1_g || !w->ln2_g) return BLK_ERR_NULL;
  if (!aligned(w->ln1_g, 16) || !aligned(w->ln2_g, 16)) return BLK_ERR_ALIGN;
  if (c.has_qkv_bias) {
    if (!w->bq || !w->bk || !w->bv) return BLK_ERR_NULL;
    if (!aligned(w->bq, 16) || !aligned(w->bk, 16) || !aligned(w->bv, 16))
      return BLK_ERR_ALIGN;
  }
  return BLK_OK;
}

// The arguments of a call other than its weights.
int check_args(blk_handle h, const void* x, const int64_t* pos, int64_t T, int64_t L,
               const void* kc, const void* vc, const void* out, const void* kn,
               const void* vn, const void* ws) {
  if (!h) return BLK_ERR_NULL;
  if (!x || !pos || !kc || !vc || !out || !ws) return BLK_ERR_NULL;
  const void* a16[] = {x, kc, vc, out, ws};
  for (const void* p : a16)
    if (!aligned(p, 16)) return BLK_ERR_ALIGN;
  if ((kn && !aligned(kn, 16)) || (vn && !aligned(vn, 16))) return BLK_ERR_ALIGN;
  if (!aligned(pos, 8)) return BLK_ERR_ALIGN;
  if (T < 1 || T > ((int64_t)1 << 31)) return BLK_ERR_SHAPE;
  if (L < 0 || L + T > h->cfg.max_ctx) return BLK_ERR_CACHE_OVERFLOW;
  return BLK_OK;
}

int check_call(blk_handle h, const blk_weights* w, const void* x,
               const int64_t* pos, int64_t T, int64_t L, const void* kc,
               const void* vc, const void* out, const void* kn, const void* vn,
               const void* ws) {
  if (!h) return BLK_ERR_NULL;
  const int rc = check_weights(h->cfg, w);
  if (rc) return rc;
  return check_args(h, x, pos, T, L, kc, vc, out, kn, vn, ws);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? BLK_OK : BLK_ERR_CUDA; }

// Brackets one launch with events when the handle's timing is on.
struct Timer {
  blk_handle h;
  cudaStream_t s;
  int slot = -1;
  void begin(int kid) {
    slot = -1;
    if (!h->timing) return;
    if (h->pending >= kMaxPending) {
      h->overflow = true;
      return;
    }
    slot = h->pending++;
    h->pending_kernel[slot] = kid;
    cudaEventRecord(h->ev[2 * slot], s);
  }
  void end() {
    if (slot >= 0) cudaEventRecord(h->ev[2 * slot + 1], s);
    slot = -1;
  }
};

#define BLK_LAUNCH(TIMER, KID, EXPR)   \
  do {                                 \
    (TIMER).begin(KID);                \
    const cudaError_t e_ = (EXPR);     \
    (TIMER).end();                     \
    if (e_ != cudaSuccess) return BLK_ERR_CUDA; \
  } while (0)

// The same tail for a decode batch of M <= kFrMaxRows rows on the few-row
// projections (gemm_fr.cu): o_proj and down write K-split partials that the
// RMSNorm 2 and the down reduction add up, gate|up applies SwiGLU itself.
int run_block_tail_few(blk_handle h, const blk_weights* w, const void* x, __half* attn16,
                       float* h32, __half* hn16, __half* act16, float* part32, int max_splits,
                       void* out, int M, cudaStream_t s, Timer& tm, const __half* next_g,
                       __half* next_xn16) {
  const blk_config& c = h->cfg;
  const int H = c.hidden, D = c.head_dim, Hq = c.n_heads, I = c.intermediate;
  FrGemmParams fo = {};
  fo.x = attn16; fo.w[0] = w->wo; fo.seg_rows[0] = H;
  fo.M = M; fo.N = H; fo.K = Hq * D;
  fo.max_splits = max_splits < kMaxSplitsNorm ? max_splits : kMaxSplitsNorm;
  fo.part = part32; fo.err = h->status;
  BLK_LAUNCH(tm, kKGemmO, launch_fr_gemm(fo, kFrPart, h->num_sms, s, true));
  BLK_LAUNCH(tm, kKRmsNorm,
             launch_rmsnorm_splitk(part32, fo.splits, static_cast<const __half*>(x), h32,
                                   static_cast<const __half*>(w->ln2_g), M, H, c.rms_eps, hn16,
                                   s, true));
  FrGemmParams fg = {};
  fg.x = hn16; fg.w[0] = w->w_gate; fg.w[1] = w->w_up;
  fg.M = M; fg.N = I; fg.K = H;
  fg.out16 = act16; fg.ldo = I; fg.err = h->status;
  BLK_LAUNCH(tm, kKGemmGateUp, launch_fr_gemm(fg, kFrGateUp, h->num_sms, s, true));
  FrGemmParams fd = {};
  fd.x = act16; fd.w[0] = w->w_down; fd.seg_rows[0] = H;
  fd.M = M; fd.N = H; fd.K = I;
  fd.max_splits = max_splits;
  fd.part = part32; fd.err = h->status;
  BLK_LAUNCH(tm, kKGemmDown, launch_fr_gemm(fd, kFrPart, h->num_sms, s, true));
  if (next_g) {
    BLK_LAUNCH(tm, kKReduceNorm,
               launch_splitk_reduce_norm(part32, fd.splits, h32, static_cast<__half*>(out),
                                         next_g, M, H, c.rms_eps, next_xn16, s));
  } else {
    TcGemmParams r = {};
    r.part = part32; r.splits = fd.splits; r.M = M; r.N = H;
    r.res32 = h32; r.out16 = static_cast<__half*>(out);
    BLK_LAUNCH(tm, kKSplitReduce, launch_splitk_reduce(r, h->num_sms, s));
  }
  return BLK_OK;
}

// o_proj + residual, RMSNorm 2, gate|up + SwiGLU, down + residual for M rows
// (shared by prefill, prefill_kv and batched decode).  With next_g set (a
// layer stack), the next layer's RMSNorm 1 of out (gain next_g) is also
// written to next_xn16, fused with the down split-K reduction when there is
// one.  few_rows (batched decode) takes the few-row projections when M is
// small enough for them.
int run_block_tail(blk_handle h, const blk_weights* w, const void* x, __half* attn16,
                   float* h32, __half* hn16, __half* act16, float* part32, int max_splits,
                   bool split_o, bool few_rows, void* out, int M, cudaStream_t s, Timer& tm,
                   const __half* next_g = nullptr, __half* next_xn16 = nullptr) {
  if (few_rows && M <= kFrMaxRows)
    return run_block_tail_few(h, w, x, attn16, h32, hn16, act16, part32, max_splits, out, M, s,
                              tm, next_g, next_xn16);
  const blk_config& c = h->cfg;
  const int H = c.hidden, D = c.head_dim, Hq = c.n_heads, I = c.intermediate;
  // o_proj + residual -> h (fp32)
  TcGemmParams go = {};
  if (make_tmap_2d(&go.tmA, attn16, M, (int64_t)Hq * D, tc_a_box_rows(M)) ||
      make_tmap_2d(&go.tmB[0], w->wo, H, (int64_t)Hq * D, 64))
    return BLK_ERR_CUDA;
  go.M = M; go.N = H; go.K = Hq * D; go.a_rows = tc_a_box_rows(M);
  go.res16 = static_cast<const __half*>(x); go.out32 = h32; go.ldo = H;
  if (split_o) {   // few rows: K splits fill the SM pairs; the partials are
    go.part = part32;   // summed (with the residual) by the RMSNorm below,
    go.max_splits = max_splits < kMaxSplitsNorm ? max_splits : kMaxSplitsNorm;   // <= 8 of them
  }
  go.err = h->status;
  BLK_LAUNCH(tm, kKGemmO, launch_tc_gemm(go, kTcResidF32, h->num_sms, s, true));

  // RMSNorm 2 (h = the o_proj partials + x when o_proj was split)
  if (go.splits > 1)
    BLK_LAUNCH(tm, kKRmsNorm,
               launch_rmsnorm_splitk(part32, go.splits, static_cast<const __half*>(x), h32,
                                     static_cast<const __half*>(w->ln2_g), M, H, c.rms_eps,
                                     hn16, s, true));
  else
    BLK_LAUNCH(tm, kKRmsNorm,
               launch_rmsnorm_rows(h32, true, static_cast<const __half*>(w->ln2_g), M, H,
                                   c.rms_eps, hn16, s, true));

  // gate | up + SwiGLU
  TcGemmParams gu = {};
  if (make_tmap_2d(&gu.tmA, hn16, M, H, tc_a_box_rows(M)) ||
      make_tmap_2d(&gu.tmB[0], w->w_gate, I, H, 64) ||
      make_tmap_2d(&gu.tmB[1], w->w_up, I, H, 64))
    return BLK_ERR_CUDA;
  gu.M = M; gu.N = I; gu.K = H; gu.a_rows = tc_a_box_rows(M);
  gu.out16 = act16; gu.ldo = I;
  gu.err = h->status;
  BLK_LAUNCH(tm, kKGemmGateUp, launch_tc_gemm(gu, kTcGateUp, h->num_sms, s, true));

  // down + residual -> out
  TcGemmParams gd = {};
  if (make_tmap_2d(&gd.tmA, act16, M, I, tc_a_box_rows(M)) ||
      make_tmap_2d(&gd.tmB[0], w->w_down, H, I, 64))
    return BLK_ERR_CUDA;
  gd.M = M; gd.N = H; gd.K = I; gd.a_rows = tc_a_box_rows(M);
  gd.res32 = h32; gd.out16 = static_cast<__half*>(out); gd.ldo = H;
  gd.part = part32;
  gd.max_splits = max_splits;
  gd.err = h->status;
  BLK_LAUNCH(tm, kKGemmDown, launch_tc_gemm(gd, kTcResidOutF16, h->num_sms, s, true));
  if (next_g && gd.splits > 1)
    BLK_LAUNCH(tm, kKReduceNorm,
               launch_splitk_reduce_norm(part32, gd.splits, h32, gd.out16, next_g, M, H,
                                         c.rms_eps, next_xn16, s));
  else if (gd.splits > 1)
    BLK_LAUNCH(tm, kKSplitReduce, launch_splitk_reduce(gd, h->num_sms, s));
  else if (next_g)
    BLK_LAUNCH(tm, kKRmsNorm,
               launch_rmsnorm_rows(out, false, next_g, M, H, c.rms_eps, next_xn16, s, true));
  return BLK_OK;
}

// prefill and prefill_kv: T new rows after L history slots.  In a layer
// stack, x_normed says that the workspace's xn16 already holds RMSNorm 1 of x
// (written by the previous layer's tail) and next_ln1, when set, has this
// layer's tail write the next layer's RMSNorm 1 there.
int run_prefill(blk_handle h, const blk_weights* w, const void* x,
                const int64_t* pos, int64_t T, int64_t L, void* k_cache,
                void* v_cache, void* out, void* k_new, void* v_new, void* ws,
                size_t ws_bytes, void* stream, bool x_normed = false,
                const __half* next_ln1 = nullptr) {
  int rc = check_call(h, w, x, pos, T, L, k_cache, v_cache, out, k_new, v_new, ws);
  if (rc) return rc;
  const blk_config& c = h->cfg;
  const PrefillWs lay = prefill_ws(c, T, h->num_sms);
  if (ws_bytes < lay.total) return BLK_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(ws);
  __half* xn16 = reinterpret_cast<__half*>(base + lay.xn16);
  __half* q16 = reinterpret_cast<__half*>(base + lay.q16);
  __half* attn16 = reinterpret_cast<__half*>(base + lay.attn16);
  float* h32 = reinterpret_cast<float*>(base + lay.h32);
  __half* hn16 = reinterpret_cast<__half*>(base + lay.hn16);
  __half* act16 = reinterpret_cast<__half*>(base + lay.act16);
  const int H = c.hidden, D = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads, M = (int)T;
  const bool first_pdl = (h->flags & BLK_FLAG_CHAIN) != 0;
  Timer tm{h, s};

  // RMSNorm 1
  if (!x_normed)
    BLK_LAUNCH(tm, kKRmsNorm,
               launch_rmsnorm_rows(x, false, static_cast<const __half*>(w->ln1_g), M, H,
                                   c.rms_eps, xn16, s, first_pdl));

  // QKV projection + bias + RoPE + KV append
  TcGemmParams g = {};
  if (make_tmap_2d(&g.tmA, xn16, M, H, tc_a_box_rows(M)) ||
      make_tmap_2d(&g.tmB[0], w->wq, (int64_t)Hq * D, H, 64) ||
      make_tmap_2d(&g.tmB[1], w->wk, (int64_t)Hkv * D, H, 64) ||
      make_tmap_2d(&g.tmB[2], w->wv, (int64_t)Hkv * D, H, 64))
    return BLK_ERR_CUDA;
  g.M = M; g.N = (Hq + 2 * Hkv) * D; g.K = H; g.a_rows = tc_a_box_rows(M);
  g.seg_rows[0] = Hq * D; g.seg_rows[1] = Hkv * D; g.seg_rows[2] = Hkv * D;
  if (c.has_qkv_bias) {
    g.bias[0] = static_cast<const __half*>(w->bq);
    g.bias[1] = static_cast<const __half*>(w->bk);
    g.bias[2] = static_cast<const __half*>(w->bv);
  }
  g.pos = pos; g.rope = h->rope; g.rope_len = c.max_ctx;
  g.Hq = Hq; g.Hkv = Hkv; g.D = D;
  g.q16 = q16;
  g.kc = static_cast<__half*>(k_cache);
  g.vc = static_cast<__half*>(v_cache);
  g.k_new = static_cast<__half*>(k_new);
  g.v_new = static_cast<__half*>(v_new);
  g.max_ctx = c.max_ctx; g.cache_len = L;
  g.err = h->status;
  // (not split in K: a split QKV projection needs qkv_finish, which costs
  // more than the split saves at T = 512, measured)
  BLK_LAUNCH(tm, kKGemmQKV, launch_tc_gemm(g, kTcQKV, h->num_sms, s, true));

  // causal GQA attention over [history; new rows]
  PrefillAttnParams pa = {};
  {
    const int64_t qd[3] = {D, Hq, M}, qs[2] = {(int64_t)D * 2, (int64_t)Hq * D * 2};
    const int qb[3] = {64, 1, 128};
    const int64_t kd[3] = {D, L + M, Hkv}, ks[2] = {(int64_t)D * 2, c.max_ctx * D * 2};
    const int kb[3] = {64, 128, 1};
    if (make_tmap_3d(&pa.tm_q, q16, qd, qs, qb) || make_tmap_3d(&pa.tm_k, k_cache, kd, ks, kb) ||
        make_tmap_3d(&pa.tm_v, v_cache, kd, ks, kb))
      return BLK_ERR_CUDA;
  }
  pa.q16 = q16;
  pa.err = h->status;
  pa.max_ctx = c.max_ctx; pa.cache_len = L;
  pa.T = M; pa.Hq = Hq; pa.Hkv = Hkv; pa.D = D;
  pa.window = h->window;
  pa.scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
  pa.attn16 = attn16;
  pa.max_chunks = prefill_attn_max_chunks(T, Hq, h->num_sms);
  pa.part = reinterpret_cast<float*>(base + lay.part32);
  plan_prefill_attn(pa, h->num_sms);
  BLK_LAUNCH(tm, kKAttnPrefill, launch_prefill_attn(pa, s, true));
  if (pa.grid_chunks > 1) BLK_LAUNCH(tm, kKAttnMerge, launch_attn_merge(pa, s, true));

  // o_proj splits K the same way when its tiles are few; the RMSNorm that
  // follows it adds the partials and the residual
  return run_block_tail(h, w, x, attn16, h32, hn16, act16,
                        reinterpret_cast<float*>(base + lay.part32), kMaxSplits, true, false,
                        out, M, s, tm, next_ln1, xn16);
}

// Batched decode: B sequences, one new token each, caches [B][Hkv][max_ctx][D].
struct DecodeBatchWs {
  size_t xn16, q16, attn16, h32, hn16, act16, part32, apart, total;
};

DecodeBatchWs decode_batch_ws(const blk_config& c, int64_t B, int num_sms) {
  const size_t H = c.hidden, D = c.head_dim, Hq = c.n_heads, I = c.intermediate;
  DecodeBatchWs w;
  size_t o = 0;
  w.xn16 = o; o = align_up(o + B * H * 2);
  w.q16 = o; o = align_up(o + B * Hq * D * 2);
  w.attn16 = o; o = align_up(o + B * Hq * D * 2);
  w.h32 = o; o = align_up(o + B * H * 4);
  w.hn16 = o; o = align_up(o + B * H * 2);
  w.act16 = o; o = align_up(o + B * I * 2);
  // split-K partials of QKV, o_proj and down (never live at the same time)
  const size_t nmax = (size_t)(Hq + 2 * c.n_kv_heads) * D > H ? (Hq + 2 * c.n_kv_heads) * D : H;
  w.part32 = o; o = align_up(o + (size_t)kMaxSplitsBatch * B * nmax * 4);
  const int smax = decode_batch_splits((int)B, c.n_kv_heads, c.max_ctx - 1, num_sms);
  w.apart = o; o = align_up(o + decode_batch_part_bytes((int)B, (int)Hq, (int)D, smax));
  w.total = o;
  return w;
}

// Every host-side check of a batched decode call (nothing is enqueued).
int check_decode_batch(blk_handle h, const blk_weights* w, const void* x, const int64_t* pos,
                       const int64_t* cache_lens, int64_t B, int64_t max_cache_len,
                       const void* k_cache, const void* v_cache, const void* out,
                       const void* k_new, const void* v_new, const void* ws, size_t ws_bytes) {
  if (!h) return BLK_ERR_NULL;
  const blk_config& c = h->cfg;
  int rc = check_weights(c, w);
  if (rc) return rc;
  if (!x || !pos || !cache_lens || !k_cache || !v_cache || !out || !ws) return BLK_ERR_NULL;
  for (const void* ptr : {x, k_cache, v_cache, out, ws})
    if (!aligned(ptr, 16)) return BLK_ERR_ALIGN;
  if (!aligned(pos, 8) || !aligned(cache_lens, 8)) return BLK_ERR_ALIGN;
  if ((k_new && !aligned(k_new, 16)) || (v_new && !aligned(v_new, 16))) return BLK_ERR_ALIGN;
  if (B < 1 || B > 4096) return BLK_ERR_SHAPE;
  if (max_cache_len < 0 || max_cache_len + 1 > c.max_ctx) return BLK_ERR_CACHE_OVERFLOW;
  if (c.n_heads / c.n_kv_heads > 16) return BLK_ERR_SHAPE;
  if (ws_bytes < decode_batch_ws(c, B, h->num_sms).total) return BLK_ERR_WORKSPACE;
  return BLK_OK;
}

// One batched-decode layer.  In a layer stack, x_normed says that the
// workspace's xn16 already holds RMSNorm 1 of x (written by the previous
// layer's tail) and next_ln1, when set, has this layer's tail write the next
// layer's RMSNorm 1 there.
int run_decode_batch(blk_handle h, const blk_weights* w, const void* x, const int64_t* pos,
                     const int64_t* cache_lens, int64_t B, int64_t max_cache_len, void* k_cache,
                     void* v_cache, void* out, void* k_new, void* v_new, void* ws,
                     size_t ws_bytes, void* stream, bool x_normed = false,
                     const __half* next_ln1 = nullptr) {
  int rc = check_decode_batch(h, w, x, pos, cache_lens, B, max_cache_len, k_cache, v_cache, out,
                              k_new, v_new, ws, ws_bytes);
  if (rc) return rc;
  const blk_config& c = h->cfg;
  const DecodeBatchWs lay = decode_batch_ws(c, B, h->num_sms);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(ws);
  __half* xn16 = reinterpret_cast<__half*>(base + lay.xn16);
  __half* q16 = reinterpret_cast<__half*>(base + lay.q16);
  __half* attn16 = reinterpret_cast<__half*>(base + lay.attn16);
  const int H = c.hidden, D = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads, M = (int)B;
  const bool first_pdl = (h->flags & BLK_FLAG_CHAIN) != 0;
  Timer tm{h, s};

  if (!x_normed)
    BLK_LAUNCH(tm, kKRmsNorm,
               launch_rmsnorm_rows(x, false, static_cast<const __half*>(w->ln1_g), M, H,
                                   c.rms_eps, xn16, s, first_pdl));

  // QKV + bias + RoPE at pos[b]; K/V to slot cache_lens[b] of sequence b's cache.
  // Up to kFrMaxRows sequences: the few-row projection writes at most 4 K-split
  // partials, which the attention kernel adds up and finishes.
  const bool few = M <= kFrMaxRows;
  FrGemmParams fq = {};
  TcGemmParams g = {};
  if (make_tmap_2d(&g.tmA, xn16, M, H, tc_a_box_rows(M)) ||
      make_tmap_2d(&g.tmB[0], w->wq, (int64_t)Hq * D, H, 64) ||
      make_tmap_2d(&g.tmB[1], w->wk, (int64_t)Hkv * D, H, 64) ||
      make_tmap_2d(&g.tmB[2], w->wv, (int64_t)Hkv * D, H, 64))
    return BLK_ERR_CUDA;
  g.M = M; g.N = (Hq + 2 * Hkv) * D; g.K = H; g.a_rows = tc_a_box_rows(M);
  g.seg_rows[0] = Hq * D; g.seg_rows[1] = Hkv * D; g.seg_rows[2] = Hkv * D;
  if (c.has_qkv_bias) {
    g.bias[0] = static_cast<const __half*>(w->bq);
    g.bias[1] = static_cast<const __half*>(w->bk);
    g.bias[2] = static_cast<const __half*>(w->bv);
  }
  g.pos = pos; g.rope = h->rope; g.rope_len = c.max_ctx;
  g.Hq = Hq; g.Hkv = Hkv; g.D = D;
  g.q16 = q16;
  g.kc = static_cast<__half*>(k_cache);
  g.vc = static_cast<__half*>(v_cache);
  g.k_new = static_cast<__half*>(k_new);
  g.v_new = static_cast<__half*>(v_new);
  g.max_ctx = c.max_ctx; g.cache_len = 0;
  g.cache_lens = cache_lens;
  g.seq_stride = (int64_t)Hkv * c.max_ctx * D;
  g.part = reinterpret_cast<float*>(base + lay.part32);   // K splits fill the SM pairs;
  g.max_splits = kMaxSplitsBatch;   // the attention kernel (or qkv_finish) applies the epilogue
  g.err = h->status;
  if (few) {
    fq.x = xn16; fq.w[0] = w->wq; fq.w[1] = w->wk; fq.w[2] = w->wv;
    for (int i = 0; i < 3; ++i) fq.seg_rows[i] = g.seg_rows[i];
    fq.M = M; fq.N = g.N; fq.K = H;
    fq.max_splits = 4;
    fq.part = g.part; fq.err = h->status;
    BLK_LAUNCH(tm, kKGemmQKV, launch_fr_gemm(fq, kFrPart, h->num_sms, s, true));
  } else {
    BLK_LAUNCH(tm, kKGemmQKV, launch_tc_gemm(g, kTcQKV, h->num_sms, s, true));
  }

  // attention of every sequence over its own slots [0, cache_lens[b]]; a
  // K-split QKV projection is finished inside it (bias, RoPE, new K/V)
  DecodeAttnBatchParams pa = {};
  const int qkv_splits = few ? fq.splits : g.splits;
  if (!few && g.splits > 4) BLK_LAUNCH(tm, kKQkvFinish, launch_qkv_finish(g, s));
  else if (few || g.splits > 1) {
    pa.qkv_part = g.part;
    pa.qkv_splits = qkv_splits;
    for (int i = 0; i < 3; ++i) pa.bias[i] = g.bias[i];
    pa.pos = pos;
    pa.rope = h->rope;
    pa.rope_len = c.max_ctx;
    pa.kc = static_cast<__half*>(k_cache);
    pa.vc = static_cast<__half*>(v_cache);
    pa.k_new = static_cast<__half*>(k_new);
    pa.v_new = static_cast<__half*>(v_new);
  }
  {
    // (64 columns, slot, D / 64 column halves, sequence x kv head): one copy
    // moves a whole 64-slot tile, [D/64][64 slots][128 B]
    const int64_t kd[4] = {64, c.max_ctx, D / 64, (int64_t)M * Hkv};
    const int64_t ks[3] = {(int64_t)D * 2, 128, c.max_ctx * D * 2};
    const int kb[4] = {64, 64, D / 64, 1};
    if (make_tmap_4d(&pa.tm_k, k_cache, kd, ks, kb) || make_tmap_4d(&pa.tm_v, v_cache, kd, ks, kb))
      return BLK_ERR_CUDA;
  }
  pa.q16 = q16;
  pa.cache_lens = cache_lens;
  pa.B = M; pa.Hq = Hq; pa.Hkv = Hkv; pa.D = D;
  pa.max_ctx = c.max_ctx;
  pa.scale_log2 = (float)(1.4426950408889634 / sqrt((double)D));
  pa.window = h->window;
  // with a window a sequence attends at most `window` slots
  pa.nsplit = decode_batch_splits(
      M, Hkv, h->window > 0 && h->window <= max_cache_len ? h->window - 1 : max_cache_len,
      h->num_sms);
  pa.deep = decode_batch_deep(M, Hkv, h->num_sms) ? 1 : 0;
  pa.part = reinterpret_cast<float*>(base + lay.apart);
  pa.attn16 = attn16;
  pa.err = h->status;
  BLK_LAUNCH(tm, kKDecodeAttnBatch, launch_decode_attn_batch(pa, s));

  return run_block_tail(h, w, x, attn16, reinterpret_cast<float*>(base + lay.h32),
                        reinterpret_cast<__half*>(base + lay.hn16),
                        reinterpret_cast<__half*>(base + lay.act16),
                        reinterpret_cast<float*>(base + lay.part32), kMaxSplitsBatch, true, true,
                        out, M, s, tm, next_ln1, xn16);
}

}  // namespace

namespace {

// ---------------------------------------------------------------- decode
// One layer's weights as the decode launch consumes them: fp16 matrices, or
// quantized codes with their scales (and int4 zero points).
struct LayerSrc {
  const void* mat[kDecRoles];   // wq wk wv wo w_gate w_up w_down
  const uint16_t* scale[kDecRoles];
  const uint8_t* zero[kDecRoles];
  const void *ln1, *ln2, *bq, *bk, *bv;
};

LayerSrc layer_src(const blk_weights& w) {
  LayerSrc s = {};
  const void* m[kDecRoles] = {w.wq, w.wk, w.wv, w.wo, w.w_gate, w.w_up, w.w_down};
  for (int r = 0; r < kDecRoles; ++r) s.mat[r] = m[r];
  s.ln1 = w.ln1_g; s.ln2 = w.ln2_g; s.bq = w.bq; s.bk = w.bk; s.bv = w.bv;
  return s;
}

LayerSrc layer_src(const blk_qweights& w) {
  LayerSrc s = {};
  const blk_qmatrix* m[kDecRoles] = {&w.wq, &w.wk, &w.wv, &w.wo, &w.w_gate, &w.w_up, &w.w_down};
  for (int r = 0; r < kDecRoles; ++r) {
    s.mat[r] = m[r]->q;
    s.scale[r] = static_cast<const uint16_t*>(m[r]->scale);
    s.zero[r] = static_cast<const uint8_t*>(m[r]->zero);
  }
  s.ln1 = w.ln1_g; s.ln2 = w.ln2_g; s.bq = w.bq; s.bk = w.bk; s.bv = w.bv;
  return s;
}

int weight_fmt(const blk_weights*) { return BLK_WFMT_F16; }
int weight_fmt(const blk_qweights* w) { return w->format; }
int weight_group(const blk_weights*) { return 0; }
int weight_group(const blk_qweights* w) { return w->group; }
int check_layer_weights(blk_handle h, const blk_weights* w) { return check_weights(h->cfg, w); }
int check_layer_weights(blk_handle h, const blk_qweights* w) { return check_qweights(h->cfg, w); }

template <typename WT>
int decode_stack_impl(blk_handle h, const WT* w, int n_layers, void* const* k_caches,
                      void* const* v_caches, const void* x, const int64_t* pos,
                      int64_t cache_len, void* out, void* const* k_new, void* const* v_new,
                      void* ws, size_t ws_bytes, void* stream) {
  if (!h || !w || !k_caches || !v_caches) return BLK_ERR_NULL;
  if (n_layers < 1) return BLK_ERR_SHAPE;
  if (!h->decode_ok) return BLK_ERR_SHAPE;
  for (int l = 0; l < n_layers; ++l) {
    int rc = check_layer_weights(h, &w[l]);
    if (rc) return rc;
    rc = check_args(h, x, pos, 1, cache_len, k_caches[l], v_caches[l], out,
                    k_new ? k_new[l] : nullptr, v_new ? v_new[l] : nullptr, ws);
    if (rc) return rc;
    if (weight_fmt(&w[l]) != weight_fmt(w) || weight_group(&w[l]) != weight_group(w))
      return BLK_ERR_SHAPE;
  }
  const blk_config& c = h->cfg;
  const int fmt = weight_fmt(w), group = weight_group(w);
  if (decode_q_max_entries(c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.intermediate, fmt,
                           group, h->num_sms) > decode_q_entry_limit())
    return BLK_ERR_SHAPE;
  if (ws_bytes < decode_ws_bytes(c.hidden, c.n_heads, c.n_kv_heads, c.head_dim,
                                 c.intermediate, h->num_sms))
    return BLK_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Timer tm{h, s};
  // DecodeParams holds the tensor maps and pointers of up to kDecMaxLayers
  // layers; it lives in the handle to keep it off the host stack.
  DecodeParams& p = *h->dec;
  for (int l0 = 0; l0 < n_layers; l0 += kDecMaxLayers) {
    const int nl = n_layers - l0 < kDecMaxLayers ? n_layers - l0 : kDecMaxLayers;
    memset(&p, 0, sizeof p);
    p.n_layers = nl;
    p.H = c.hidden; p.Hq = c.n_heads; p.Hkv = c.n_kv_heads; p.D = c.head_dim;
    p.I = c.intermediate; p.eps = c.rms_eps;
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
    p.max_ctx = c.max_ctx; p.cache_len = cache_len; p.pos = pos;
    p.rope = h->rope; p.rope_len = c.max_ctx;
    p.x_in = static_cast<const __half*>(l0 == 0 ? x : out);
    p.out = static_cast<__half*>(out);
    p.err = h->status;
    p.trace = h->trace;
    p.trace_len = h->trace_len;
    p.fmt = fmt;
    p.qgroup = group;
    p.qgroup_lg = 0;
    while (group > 0 && (1 << p.qgroup_lg) < group) ++p.qgroup_lg;
    p.window = h->window;
    decode_ws_carve(p, ws, h->num_sms);
    for (int k = 0; k < nl; ++k) {
      const LayerSrc src = layer_src(w[l0 + k]);
      DecLayer& d = p.layer[k];
      d.wq = static_cast<const __half*>(src.mat[0]);
      d.wk = static_cast<const __half*>(src.mat[1]);
      d.wv = static_cast<const __half*>(src.mat[2]);
      if (c.has_qkv_bias) {
        d.bq = static_cast<const __half*>(src.bq);
        d.bk = static_cast<const __half*>(src.bk);
        d.bv = static_cast<const __half*>(src.bv);
      }
      d.wo = static_cast<const __half*>(src.mat[3]);
      d.ln1 = static_cast<const __half*>(src.ln1);
      d.ln2 = static_cast<const __half*>(src.ln2);
      d.wg = static_cast<const __half*>(src.mat[4]);
      d.wu = static_cast<const __half*>(src.mat[5]);
      d.wd = static_cast<const __half*>(src.mat[6]);
      d.kc = static_cast<__half*>(k_caches[l0 + k]);
      d.vc = static_cast<__half*>(v_caches[l0 + k]);
      d.k_new = static_cast<__half*>(k_new ? k_new[l0 + k] : nullptr);
      d.v_new = static_cast<__half*>(v_new ? v_new[l0 + k] : nullptr);
      const int64_t rows = (int64_t)c.n_kv_heads * c.max_ctx;
      if (make_tmap_2d(&p.tm_k[k], d.kc, rows, c.head_dim, 64) ||
          make_tmap_2d(&p.tm_v[k], d.vc, rows, c.head_dim, 64))
        return BLK_ERR_CUDA;
      // weights as 8-row boxes: {rows, K} per role
      const int64_t H = c.hidden, QD = (int64_t)c.n_heads * c.head_dim,
                    KD = (int64_t)c.n_kv_heads * c.head_dim, I = c.intermediate;
      const int64_t rk[kDecRoles][2] = {{QD, H}, {KD, H}, {KD, H}, {H, QD},
                                        {I, H},  {I, H},  {H, I}};
      for (int r = 0; r < kDecRoles; ++r) {
        int is3d = 0;
        if (fmt == BLK_WFMT_F16) {
          const int64_t nz = (rk[r][1] + 63) / 64;
          const int cbs = (int)(nz < 24 ? nz : 24);
          if (make_tmap_rows8(&p.tm_w[k][r], src.mat[r], rk[r][0], rk[r][1], cbs, &is3d))
            return BLK_ERR_CUDA;
          p.wbox_z[r] = cbs;
          p.wnz[r] = (int)nz;
        } else {
          // code bytes per row; a box row covers 12 blocks of 128 INT8 codes
          // or 6 blocks of 256 int4 codes: 1536 columns either way
          const int64_t row_bytes = fmt == BLK_WFMT_I8 ? rk[r][1] : rk[r][1] / 2;
          const int64_t nz = (row_bytes + 127) / 128;
          const int per = fmt == BLK_WFMT_I8 ? 12 : 6;
          const int cbs = (int)(nz < per ? nz : per);
          if (make_tmap_codes(&p.tm_w[k][r], src.mat[r], rk[r][0], row_bytes, cbs, &is3d))
            return BLK_ERR_CUDA;
          p.wbox_z[r] = cbs;
          p.wnz[r] = (int)nz;
          p.qscale[k][r] = src.scale[r];
          p.qzero[k][r] = src.zero[r];
        }
        p.w3d[r] = is3d;
      }
    }
    BLK_LAUNCH(tm, kKDecodeStep, launch_decode_persistent(p, h->num_sms, s));
  }
  return BLK_OK;
}

// ------------------------------------------------------ quantized prefill
size_t layer_f16_bytes(const blk_config& c) {
  const size_t H = c.hidden, QD = (size_t)c.n_heads * c.head_dim,
               KD = (size_t)c.n_kv_heads * c.head_dim, I = c.intermediate;
  return 2 * (QD * H + 2 * KD * H + H * QD + 3 * I * H) + 7 * kAlign;
}

// Forms the layer's weights as fp16 at the start of the workspace, then runs
// the fp16 prefill on them with the rest of the workspace.
int run_prefill_q(blk_handle h, const blk_qweights* w, const void* x, const int64_t* pos,
                  int64_t T, int64_t L, void* k_cache, void* v_cache, void* out, void* k_new,
                  void* v_new, void* ws, size_t ws_bytes, void* stream) {
  if (!h) return BLK_ERR_NULL;
  int rc = check_qweights(h->cfg, w);
  if (rc) return rc;
  rc = check_args(h, x, pos, T, L, k_cache, v_cache, out, k_new, v_new, ws);
  if (rc) return rc;
  const blk_config& c = h->cfg;
  const size_t wbytes = align_up(layer_f16_bytes(c));
  if (ws_bytes < wbytes) return BLK_ERR_WORKSPACE;
  if (ws_bytes - wbytes < prefill_ws(c, T, h->num_sms).total) return BLK_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t H = c.hidden, QD = (int64_t)c.n_heads * c.head_dim,
                KD = (int64_t)c.n_kv_heads * c.head_dim, I = c.intermediate;
  const blk_qmatrix* m[kDecRoles] = {&w->wq, &w->wk, &w->wv, &w->wo, &w->w_gate, &w->w_up,
                                     &w->w_down};
  const int64_t rk[kDecRoles][2] = {{QD, H}, {KD, H}, {KD, H}, {H, QD}, {I, H}, {I, H}, {H, I}};
  unsigned char* base = static_cast<unsigned char*>(ws);
  __half* f16[kDecRoles];
  size_t o = 0;
  for (int r = 0; r < kDecRoles; ++r) {
    f16[r] = reinterpret_cast<__half*>(base + o);
    o = align_up(o + (size_t)rk[r][0] * rk[r][1] * 2);
  }
  {
    Timer tm{h, s};
    for (int r = 0; r < kDecRoles; ++r)
      BLK_LAUNCH(tm, kKDequant, launch_dequant(w->format, m[r]->q, m[r]->scale, m[r]->zero,
                                               rk[r][0], rk[r][1], w->group, f16[r],
                                               h->num_sms, s));
  }
  blk_weights fw = {};
  fw.ln1_g = w->ln1_g; fw.ln2_g = w->ln2_g; fw.bq = w->bq; fw.bk = w->bk; fw.bv = w->bv;
  fw.wq = f16[0]; fw.wk = f16[1]; fw.wv = f16[2]; fw.wo = f16[3];
  fw.w_gate = f16[4]; fw.w_up = f16[5]; fw.w_down = f16[6];
  // the dequantized weights were written by the kernels just enqueued: the
  // first prefill kernel must not start early (no chained launch here)
  const uint32_t flags = h->flags;
  h->flags &= ~BLK_FLAG_CHAIN;
  rc = run_prefill(h, &fw, x, pos, T, L, k_cache, v_cache, out, k_new, v_new, base + wbytes,
                   ws_bytes - wbytes, stream);
  h->flags = flags;
  return rc;
}

}  // namespace

extern "C" {

// The handle's rotation table [max_ctx][head_dim / 2] of (cos, sin) pairs,
// computed in f64 and stored as fp32.  Plain RoPE: pair i of position p turns
// by p * theta^(-2i / D).  YaRN (y != NULL; the ds4.c study notes, Part 4,
// "Trace 1: YaRN frequency scaling" and the tail-rotation listing): the
// notes' ramp 1 - clamp((i - low) / max(0.001, high - low), 0, 1) between
// low = corr_dim(beta_fast) and high = corr_dim(beta_slow), corr_dim(n) =
// D ln(n_ctx_orig / (2 pi n)) / (2 ln theta); the angle blends the
// interpolated freq_scale * a and the original a with weight ramp *
// ext_factor on the original; cos and sin are scaled by attn_factor * (1 +
// 0.1 ln(1 / freq_scale)) when ext_factor != 0 (else attn_factor), the YaRN
// method's temperature, so q . k carries it squared.
static void rope_table(const blk_config& c, const blk_yarn* y, std::vector<float2>& table) {
  const int half = c.head_dim / 2;
  const double D = (double)c.head_dim, theta = (double)c.rope_theta;
  table.assign((size_t)c.max_ctx * half, make_float2(0.f, 0.f));
  const double pi = 3.14159265358979323846;
  auto corr_dim = [&](double n_rot) {
    return D * log((double)y->n_ctx_orig / (n_rot * 2.0 * pi)) / (2.0 * log(theta));
  };
  const double low = y ? corr_dim(y->beta_fast) : 0.0, high = y ? corr_dim(y->beta_slow) : 0.0;
  const double m = !y ? 1.0
                      : (y->ext_factor != 0.0
                             ? y->attn_factor * (1.0 + 0.1 * log(1.0 / y->freq_scale))
                             : y->attn_factor);
  for (int i = 0; i < half; ++i) {
    const double inv = pow(theta, -2.0 * i / D);
    double r = 0.0;   // weight of the original frequency
    if (y) {
      const double t = ((double)i - low) / (high - low > 0.001 ? high - low : 0.001);
      r = (1.0 - (t < 0.0 ? 0.0 : (t > 1.0 ? 1.0 : t))) * y->ext_factor;
    }
    for (int64_t p = 0; p < c.max_ctx; ++p) {
      const double a_orig = (double)p * inv;
      const double a = y ? (y->freq_scale * a_orig) * (1.0 - r) + a_orig * r : a_orig;
      table[(size_t)p * half + i] = make_float2((float)(cos(a) * m), (float)(sin(a) * m));
    }
  }
}

int blk_create(const blk_config* cfg, blk_handle* out) {
  if (!cfg || !out) return BLK_ERR_NULL;
  *out = nullptr;
  int rc = shape_ok(cfg);
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BLK_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return BLK_ERR_CUDA;
  if (major != 10 || minor != 3) return BLK_ERR_DEVICE;
  if (configure_kernels() != cudaSuccess) return BLK_ERR_CUDA;

  blk_handle h = new (std::nothrow) blk_handle_s();
  if (!h) return BLK_ERR_CUDA;
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = sms;
  {
    // the decode kernel stages at most kDecMaxVec inputs and keeps the
    // residual of at most 152 o_proj rows (8-row units) per CTA (one per SM)
    const int64_t rows_o = 8 * ((cfg->hidden / 8 + sms - 1) / sms);
    h->decode_ok = cfg->hidden <= kDecMaxVec && cfg->intermediate <= kDecMaxVec &&
                   cfg->n_heads * cfg->head_dim <= kDecMaxVec && cfg->n_kv_heads <= sms &&
                   cfg->n_heads / cfg->n_kv_heads <= 16 && rows_o <= 152 &&
                   cfg->intermediate % 16 == 0;
  }
  h->dec = new (std::nothrow) blk::DecodeParams();
  if (!h->dec) {
    delete h;
    return BLK_ERR_CUDA;
  }

  std::vector<float2> table;
  rope_table(*cfg, nullptr, table);
  if (cudaMalloc(&h->rope, table.size() * sizeof(float2)) != cudaSuccess ||
      cudaMalloc(&h->status, sizeof(int)) != cudaSuccess ||
      cudaMemcpy(h->rope, table.data(), table.size() * sizeof(float2),
                 cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) {
    blk_destroy(h);
    return BLK_ERR_CUDA;
  }
  *out = h;
  return BLK_OK;
}

void blk_destroy(blk_handle h) {
  if (!h) return;
  if (h->rope) cudaFree(h->rope);
  if (h->status) cudaFree(h->status);
  if (h->ev) {
    for (int i = 0; i < 2 * kMaxPending; ++i) cudaEventDestroy(h->ev[i]);
    delete[] h->ev;
  }
  delete h->dec;
  delete h;
}

int blk_set_flags(blk_handle h, uint32_t flags) {
  if (!h) return BLK_ERR_NULL;
  h->flags = flags;
  return BLK_OK;
}

int blk_set_window(blk_handle h, int64_t window) {
  if (!h) return BLK_ERR_NULL;
  if (window < 0) return BLK_ERR_SHAPE;
  h->window = window;
  return BLK_OK;
}

int blk_set_rope_yarn(blk_handle h, const blk_yarn* y) {
  if (!h) return BLK_ERR_NULL;
  if (y && !(y->freq_scale > 0.0 && y->freq_scale <= 1.0 && y->ext_factor >= 0.0 &&
             y->ext_factor <= 1.0 && y->attn_factor > 0.0 && y->beta_fast > 0.0 &&
             y->beta_slow > 0.0 && y->n_ctx_orig >= 1))
    return BLK_ERR_SHAPE;
  std::vector<float2> table;
  rope_table(h->cfg, y, table);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return BLK_ERR_CUDA;
  // the table is read by kernels already enqueued: let them finish first
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(h->rope, table.data(), table.size() * sizeof(float2),
                 cudaMemcpyHostToDevice) != cudaSuccess)
    return BLK_ERR_CUDA;
  return BLK_OK;
}

size_t blk_workspace_bytes(blk_handle h, int64_t max_T) {
  if (!h || max_T < 1) return 0;
  const blk_config& c = h->cfg;
  // Enough for every T <= max_T: the attention's chunk partials shrink at
  // some row-block counts, so take the largest layout over the T that end a
  // 128-row block (within one block the other buffers only grow with T).
  size_t a = prefill_ws(c, max_T, h->num_sms).total;
  for (int64_t t = 128; t < max_T; t += 128) {
    const size_t at = prefill_ws(c, t, h->num_sms).total;
    if (at > a) a = at;
  }
  const size_t b = decode_ws_bytes(c.hidden, c.n_heads, c.n_kv_heads, c.head_dim,
                                   c.intermediate, h->num_sms);
  return a > b ? a : b;
}

int blk_prefill(blk_handle h, const blk_weights* w, const void* x,
                const int64_t* pos, int64_t T, void* k_cache, void* v_cache,
                void* out, void* k_new, void* v_new, void* ws, size_t ws_bytes,
                void* stream) {
  return run_prefill(h, w, x, pos, T, 0, k_cache, v_cache, out, k_new, v_new, ws,
                     ws_bytes, stream);
}

int blk_prefill_kv(blk_handle h, const blk_weights* w, const void* x,
                   const int64_t* pos, int64_t T, int64_t cache_len,
                   void* k_cache, void* v_cache, void* out, void* k_new,
                   void* v_new, void* ws, size_t ws_bytes, void* stream) {
  return run_prefill(h, w, x, pos, T, cache_len, k_cache, v_cache, out, k_new,
                     v_new, ws, ws_bytes, stream);
}

size_t blk_prefill_stack_workspace_bytes(blk_handle h, int64_t max_T) {
  const size_t one = blk_workspace_bytes(h, max_T);
  if (!one) return 0;
  return one + 2 * align_up((size_t)max_T * h->cfg.hidden * 2);
}

int blk_prefill_stack(blk_handle h, const blk_weights* w, int n_layers, void* const* k_caches,
                      void* const* v_caches, const void* x, const int64_t* pos, int64_t T,
                      int64_t cache_len, void* out, void* ws, size_t ws_bytes, void* stream) {
  if (!h || !w || !k_caches || !v_caches || !ws) return BLK_ERR_NULL;
  if (n_layers < 1 || T < 1) return BLK_ERR_SHAPE;
  // the two activation buffers between layers follow the one-layer workspace
  const size_t act = align_up((size_t)T * h->cfg.hidden * 2);
  const size_t layer_ws = prefill_ws(h->cfg, T, h->num_sms).total;
  if (ws_bytes < layer_ws + 2 * act) return BLK_ERR_WORKSPACE;
  unsigned char* base = static_cast<unsigned char*>(ws);
  void* bufs[2] = {base + layer_ws, base + layer_ws + act};
  auto layer_in = [&](int l) -> const void* { return l == 0 ? x : bufs[(l - 1) % 2]; };
  auto layer_out = [&](int l) -> void* { return l == n_layers - 1 ? out : bufs[l % 2]; };
  // every layer's arguments are checked before anything is enqueued
  for (int l = 0; l < n_layers; ++l) {
    const int rc = check_call(h, &w[l], layer_in(l), pos, T, cache_len, k_caches[l],
                              v_caches[l], layer_out(l), nullptr, nullptr, ws);
    if (rc) return rc;
  }
  for (int l = 0; l < n_layers; ++l) {
    // layer l's tail writes layer l + 1's RMSNorm 1 (one launch fewer a layer)
    const __half* next_ln1 =
        l + 1 < n_layers ? static_cast<const __half*>(w[l + 1].ln1_g) : nullptr;
    const int rc = run_prefill(h, &w[l], layer_in(l), pos, T, cache_len, k_caches[l],
                               v_caches[l], layer_out(l), nullptr, nullptr, ws, layer_ws, stream,
                               l > 0, next_ln1);
    if (rc) return rc;
  }
  return BLK_OK;
}

int blk_decode(blk_handle h, const blk_weights* w, const void* x,
               const int64_t* pos, int64_t cache_len, void* k_cache,
               void* v_cache, void* out, void* k_new, void* v_new, void* ws,
               size_t ws_bytes, void* stream) {
  void* kcs[1] = {k_cache};
  void* vcs[1] = {v_cache};
  void* kns[1] = {k_new};
  void* vns[1] = {v_new};
  return blk_decode_stack(h, w, 1, kcs, vcs, x, pos, cache_len, out, kns, vns, ws, ws_bytes,
                          stream);
}

int blk_decode_stack(blk_handle h, const blk_weights* w, int n_layers,
                     void* const* k_caches, void* const* v_caches, const void* x,
                     const int64_t* pos, int64_t cache_len, void* out,
                     void* const* k_new, void* const* v_new, void* ws, size_t ws_bytes,
                     void* stream) {
  return decode_stack_impl(h, w, n_layers, k_caches, v_caches, x, pos, cache_len, out, k_new,
                           v_new, ws, ws_bytes, stream);
}

int blk_decode_stack_q(blk_handle h, const blk_qweights* w, int n_layers,
                       void* const* k_caches, void* const* v_caches, const void* x,
                       const int64_t* pos, int64_t cache_len, void* out, void* const* k_new,
                       void* const* v_new, void* ws, size_t ws_bytes, void* stream) {
  return decode_stack_impl(h, w, n_layers, k_caches, v_caches, x, pos, cache_len, out, k_new,
                           v_new, ws, ws_bytes, stream);
}

int blk_decode_q(blk_handle h, const blk_qweights* w, const void* x, const int64_t* pos,
                 int64_t cache_len, void* k_cache, void* v_cache, void* out, void* k_new,
                 void* v_new, void* ws, size_t ws_bytes, void* stream) {
  void* kcs[1] = {k_cache};
  void* vcs[1] = {v_cache};
  void* kns[1] = {k_new};
  void* vns[1] = {v_new};
  return decode_stack_impl(h, w, 1, kcs, vcs, x, pos, cache_len, out, kns, vns, ws, ws_bytes,
                           stream);
}

size_t blk_qworkspace_bytes(blk_handle h, int64_t max_T) {
  if (!h || max_T < 1) return 0;
  return align_up(layer_f16_bytes(h->cfg)) + blk_workspace_bytes(h, max_T);
}

int blk_prefill_q(blk_handle h, const blk_qweights* w, const void* x, const int64_t* pos,
                  int64_t T, void* k_cache, void* v_cache, void* out, void* k_new, void* v_new,
                  void* ws, size_t ws_bytes, void* stream) {
  return run_prefill_q(h, w, x, pos, T, 0, k_cache, v_cache, out, k_new, v_new, ws, ws_bytes,
                       stream);
}

int blk_prefill_kv_q(blk_handle h, const blk_qweights* w, const void* x, const int64_t* pos,
                     int64_t T, int64_t cache_len, void* k_cache, void* v_cache, void* out,
                     void* k_new, void* v_new, void* ws, size_t ws_bytes, void* stream) {
  return run_prefill_q(h, w, x, pos, T, cache_len, k_cache, v_cache, out, k_new, v_new, ws,
                       ws_bytes, stream);
}

}  // extern "C"

namespace {
// Polls *flag until it is non-zero or limit_ns of %globaltimer have passed;
// a timeout records kDevTimeout in the status word, as every kernel's own
// bounded waits do.
__global__ void wait_probe_kernel(const volatile int* flag, uint64_t limit_ns, int* err) {
  const uint64_t t0 = global_ns();
  while (*flag == 0) {
    if (global_ns() - t0 > limit_ns) {
      set_error(err, kDevTimeout);
      return;
    }
  }
}
}  // namespace

extern "C" {

int blk_wait_probe(blk_handle h, const void* flag, uint64_t limit_ns, void* stream) {
  if (!h || !flag) return BLK_ERR_NULL;
  if (!aligned(flag, 4)) return BLK_ERR_ALIGN;
  if (limit_ns < 1000 || limit_ns > 2000000000ull) return BLK_ERR_SHAPE;
  wait_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const volatile int*>(flag), limit_ns, h->status);
  return cudaGetLastError() == cudaSuccess ? BLK_OK : BLK_ERR_CUDA;
}

int blk_check(blk_handle h, void* stream) {
  if (!h) return BLK_ERR_NULL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BLK_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return BLK_ERR_CUDA;
  if (v != 0 && cudaMemset(h->status, 0, sizeof v) != cudaSuccess) return BLK_ERR_CUDA;
  if (v == kDevTimeout) return BLK_ERR_DEVICE_TIMEOUT;
  if (v == kDevPosition) return BLK_ERR_POSITION;
  if (v == kDevToken) return BLK_ERR_TOKEN;
  return BLK_OK;
}

int blk_embed(blk_handle h, const void* table, int64_t vocab, const int64_t* ids, int64_t T,
              void* x, void* stream) {
  if (!h) return BLK_ERR_NULL;
  if (!table || !ids || !x) return BLK_ERR_NULL;
  if (!aligned(table, 16) || !aligned(x, 16) || !aligned(ids, 8)) return BLK_ERR_ALIGN;
  if (T <= 0 || T > (1 << 20) || vocab <= 0) return BLK_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Timer tm{h, s};
  BLK_LAUNCH(tm, kKEmbed,
             launch_embed(static_cast<const __half*>(table), vocab, ids, (int)T, h->cfg.hidden,
                          static_cast<__half*>(x), h->status, s,
                          (h->flags & BLK_FLAG_CHAIN) != 0));
  return BLK_OK;
}

size_t blk_lm_head_workspace_bytes(blk_handle h) {
  if (!h) return 0;
  return lm_head_workspace_bytes(h->num_sms);
}

int blk_lm_head(blk_handle h, const void* x, int64_t T, const void* norm_g, const void* w_lm,
                int64_t vocab, float* logits, int64_t* tokens, void* ws, size_t ws_bytes,
                void* stream) {
  if (!h) return BLK_ERR_NULL;
  if (!x || !norm_g || !w_lm || !tokens || !ws) return BLK_ERR_NULL;
  if (!aligned(x, 16) || !aligned(w_lm, 16) || !aligned(norm_g, 16) || !aligned(tokens, 8) ||
      !aligned(ws, 16) || (logits && !aligned(logits, 4)))
    return BLK_ERR_ALIGN;
  const int H = h->cfg.hidden;
  if (T < 1 || T > 8 || vocab < 1 || vocab > ((int64_t)1 << 31) - 16 || H > 4096)
    return BLK_ERR_SHAPE;
  if (ws_bytes < lm_head_workspace_bytes(h->num_sms)) return BLK_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LmHeadParams p = {};
  {
    const int64_t dims[3] = {64, vocab, H / 64}, strides[2] = {(int64_t)H * 2, 128};
    // always 24 column blocks (48 KB per copy; blocks past H arrive as zeros)
    const int box[3] = {64, 16, 24};
    if (make_tmap_3d(&p.tm_w, w_lm, dims, strides, box)) return BLK_ERR_CUDA;
  }
  p.x = static_cast<const __half*>(x);
  p.g = static_cast<const __half*>(norm_g);
  p.eps = h->cfg.rms_eps;
  p.T = (int)T;
  p.H = H;
  p.vocab = vocab;
  p.logits = logits;
  p.part_v = static_cast<float*>(ws);
  p.part_i = reinterpret_cast<int*>(static_cast<unsigned char*>(ws) +
                                    (size_t)h->num_sms * 8 * sizeof(float));
  p.token = tokens;
  p.err = h->status;
  Timer tm{h, s};
  BLK_LAUNCH(tm, kKLmHead, launch_lm_head(p, h->num_sms, s, (h->flags & BLK_FLAG_CHAIN) != 0));
  BLK_LAUNCH(tm, kKArgmax, launch_argmax_reduce(p, s));
  return BLK_OK;
}

// Largest batched-decode layout over B' <= max_B (the attention's split
// partials, B' x splits(B'), do not grow monotonically with B').
static size_t decode_batch_ws_upto(const blk_config& c, int64_t max_B, int num_sms) {
  size_t best = 0;
  for (int64_t b = 1; b <= max_B; ++b) {
    const size_t t = decode_batch_ws(c, b, num_sms).total;
    if (t > best) best = t;
  }
  return best;
}

size_t blk_decode_batch_workspace_bytes(blk_handle h, int64_t max_B) {
  if (!h || max_B < 1 || max_B > 4096) return 0;
  return decode_batch_ws_upto(h->cfg, max_B, h->num_sms);
}

int blk_decode_batch(blk_handle h, const blk_weights* w, const void* x, const int64_t* pos,
                     const int64_t* cache_lens, int64_t B, int64_t max_cache_len, void* k_cache,
                     void* v_cache, void* out, void* k_new, void* v_new, void* ws,
                     size_t ws_bytes, void* stream) {
  return run_decode_batch(h, w, x, pos, cache_lens, B, max_cache_len, k_cache, v_cache, out,
                          k_new, v_new, ws, ws_bytes, stream);
}

size_t blk_decode_batch_stack_workspace_bytes(blk_handle h, int64_t max_B) {
  if (!h || max_B < 1 || max_B > 4096) return 0;
  const size_t act = align_up((size_t)max_B * h->cfg.hidden * 2);
  return decode_batch_ws_upto(h->cfg, max_B, h->num_sms) + 2 * act;
}

int blk_decode_batch_stack(blk_handle h, const blk_weights* w, int n_layers,
                           void* const* k_caches, void* const* v_caches, const void* x,
                           const int64_t* pos, const int64_t* cache_lens, int64_t B,
                           int64_t max_cache_len, void* out, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!h || !w || !k_caches || !v_caches || !ws) return BLK_ERR_NULL;
  if (n_layers < 1 || B < 1 || B > 4096) return BLK_ERR_SHAPE;
  // the two activation buffers between layers follow the one-layer workspace
  const size_t act = align_up((size_t)B * h->cfg.hidden * 2);
  const size_t layer_ws = decode_batch_ws(h->cfg, B, h->num_sms).total;
  if (ws_bytes < layer_ws + 2 * act) return BLK_ERR_WORKSPACE;
  unsigned char* base = static_cast<unsigned char*>(ws);
  void* bufs[2] = {base + layer_ws, base + layer_ws + act};
  auto layer_in = [&](int l) -> const void* { return l == 0 ? x : bufs[(l - 1) % 2]; };
  auto layer_out = [&](int l) -> void* { return l == n_layers - 1 ? out : bufs[l % 2]; };
  // every layer's arguments are checked before anything is enqueued
  for (int l = 0; l < n_layers; ++l) {
    const int rc = check_decode_batch(h, &w[l], layer_in(l), pos, cache_lens, B, max_cache_len,
                                      k_caches[l], v_caches[l], layer_out(l), nullptr, nullptr,
                                      ws, layer_ws);
    if (rc) return rc;
  }
  for (int l = 0; l < n_layers; ++l) {
    // layer l's tail writes layer l + 1's RMSNorm 1 (one launch fewer a layer)
    const __half* next_ln1 =
        l + 1 < n_layers ? static_cast<const __half*>(w[l + 1].ln1_g) : nullptr;
    const int rc = run_decode_batch(h, &w[l], layer_in(l), pos, cache_lens, B, max_cache_len,
                                    k_caches[l], v_caches[l], layer_out(l), nullptr, nullptr, ws,
                                    layer_ws, stream, l > 0, next_ln1);
    if (rc) return rc;
  }
  return BLK_OK;
}

}  // extern "C"

size_t blk_internal_decode_ws_bytes(blk_handle h) {
  const blk_config& c = h->cfg;
  return decode_ws_bytes(c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.intermediate,
                         h->num_sms);
}

int blk_internal_device(blk_handle h) { return h->device; }

extern "C" {

int blk_set_trace(blk_handle h, void* device_buffer, size_t bytes) {
  if (!h) return BLK_ERR_NULL;
  h->trace = static_cast<uint64_t*>(device_buffer);
  h->trace_len = device_buffer ? bytes / sizeof(uint64_t) : 0;
  return BLK_OK;
}

int blk_timing(blk_handle h, int on) {
  if (!h) return BLK_ERR_NULL;
  if (on && !h->ev) {
    h->ev = new (std::nothrow) cudaEvent_t[2 * kMaxPending]();
    if (!h->ev) return BLK_ERR_CUDA;
    for (int i = 0; i < 2 * kMaxPending; ++i)
      if (cudaEventCreate(&h->ev[i]) != cudaSuccess) return BLK_ERR_CUDA;
  }
  h->timing = on != 0;
  return BLK_OK;
}

int blk_timing_collect(blk_handle h, void* stream) {
  if (!h) return BLK_ERR_NULL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BLK_ERR_CUDA;
  for (int i = 0; i < h->pending; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, h->ev[2 * i], h->ev[2 * i + 1]) != cudaSuccess)
      return BLK_ERR_CUDA;
    h->total_ms[h->pending_kernel[i]] += ms;
    h->launches[h->pending_kernel[i]] += 1;
  }
  h->pending = 0;
  const bool over = h->overflow;
  h->overflow = false;
  return over ? BLK_ERR_WORKSPACE : BLK_OK;
}

int blk_timing_read(blk_handle h, int kernel, double* total_ms, int64_t* launches,
                    const char** name) {
  if (!h) return BLK_ERR_NULL;
  if (kernel < 0 || kernel >= kKCount) return BLK_ERR_SHAPE;
  if (total_ms) *total_ms = h->total_ms[kernel];
  if (launches) *launches = h->launches[kernel];
  if (name) *name = kKernelNames[kernel];
  return BLK_OK;
}

const char* blk_status_str(int status) {
  switch (status) {
    case BLK_OK: return "ok";
    case BLK_ERR_NULL: return "a required pointer is NULL";
    case BLK_ERR_ALIGN: return "a pointer is not aligned (16 bytes for tensors, 8 for position ids)";
    case BLK_ERR_SHAPE: return "unsupported or inconsistent shape";
    case BLK_ERR_CACHE_OVERFLOW: return "cache_len + T exceeds max_ctx (or cache_len < 0)";
    case BLK_ERR_WORKSPACE: return "workspace smaller than blk_workspace_bytes()";
    case BLK_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case BLK_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case BLK_ERR_POSITION: return "a position id was outside [0, max_ctx) and was clamped";
    case BLK_ERR_TOKEN: return "a token id was outside [0, vocab) (embedding row zeroed)";
    case BLK_ERR_DEVICE: return "the current GPU is not sm_103 (GB300)";
    case BLK_ERR_SCRATCH_LIMIT:
      return "the shape needs more decode scratch than blk_decode_static's fixed 1 MiB array";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace blk {
cudaError_t configure_kernels() {
  cudaError_t e = configure_decode_persistent();
  if (e == cudaSuccess) e = configure_tc_gemm_kernels();
  if (e == cudaSuccess) e = configure_fr_gemm_kernels();
  if (e == cudaSuccess) e = configure_prefill_attn();
  if (e == cudaSuccess) e = configure_lm_head();
  if (e == cudaSuccess) e = configure_decode_attn_batch();
  return e;
}
}  // namespace blk
