/*
 * CPU oracle for one Qwen2-style decoder block — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * this library.  The GPU library never links, includes or calls it, and it
 * never calls the GPU library: the two share no code.
 *
 * Everything is plain, single-threaded C++ with f64 arithmetic.  fp16 values
 * (IEEE binary16, passed as raw uint16_t bit patterns) are decoded exactly to
 * f64; the only roundings to fp16 are the K/V written to the cache and the
 * block output, both round-to-nearest-even.
 *
 * Block definition followed (web page "An MLIR-based LLM compilation method",
 * TopOp/TpuOp paper translation, §3.1 Listings 1 and 2; §4.1 for the three
 * phases): RMSNorm -> q/k/v MatMul -> Gather cos/sin by position_ids -> Rope
 * on q and k -> (Concat with history K/V) -> FAttention -> o MatMul + input ->
 * RMSNorm -> MLP + residual -> return (o, k, v).
 *
 * Readings where the page is silent (each also listed in the design notes):
 *   RMSNorm   y_i = x_i / sqrt(mean(x^2) + eps) * g_i
 *   Rope      rotate_half pairs (i, i + D/2), angle = pos * theta^(-2i/D)
 *   FAttention softmax(q.k / sqrt(D)) over slots 0 .. L+t (causal, slot order),
 *             q head h reads kv head h / (Hq/Hkv)
 *   MLP       SwiGLU: down(silu(gate(x)) * up(x)), silu(z) = z / (1 + e^-z)
 *   biases    q/k/v only, and only when has_qkv_bias
 *   returned K is after Rope, V as projected; both also land in cache slots
 *   [L, L+T).
 *
 * Parity status of each function (what pins it without trusting itself) is
 * given beside it; the full-size block output is pinned only through the
 * component pins and the small-case brute-force checks ("parity unpinned by
 * the pages": they print no worked numeric example).
 */
#ifndef BLK_ORACLE_H
#define BLK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* YaRN RoPE (the ds4.c study notes, Part 4, "Trace 1: YaRN frequency
 * scaling" and "Trace 2: RoPE tail rotation").  The notes give the ramp, the
 * correction dimension and the per-layer scale; they elide how the ramp
 * blends the original and the scaled frequency and never define the
 * magnitude factor.  Readings (also in the design notes), from the YaRN
 * method the notes trace ("NTK-by-parts" interpolation plus an attention
 * temperature):
 *   low  = corr_dim(beta_fast), high = corr_dim(beta_slow) (no rounding)
 *   frequency pair i (rotate_half partners i, i + D/2; the ramp's i0 = 2i):
 *     a_orig = pos * theta^(-2i/D),  a_int = freq_scale * a_orig,
 *     r = ramp(low, high, 2i) * ext_factor,
 *     angle = a_int * (1 - r) + a_orig * r
 *   magnitude m = attn_factor * (1 + 0.1 ln(1 / freq_scale)) when
 *     ext_factor != 0, else attn_factor; both cos and sin are scaled by m. */
typedef struct {
  double freq_scale;    /* 1/s: the interpolated frequencies are s times lower */
  double ext_factor;    /* weight of the ramp (the notes: 1 on scaled layers, else 0) */
  double attn_factor;   /* extra magnitude factor (1 = none) */
  double beta_fast;     /* rotations over the original context that start the ramp */
  double beta_slow;     /* ... and end it */
  int64_t n_ctx_orig;   /* the original training context */
} orc_yarn;

typedef struct {
  int64_t hidden, n_heads, n_kv_heads, head_dim, intermediate;
  double rms_eps, rope_theta;
  int64_t max_ctx;
  int64_t has_qkv_bias;
  /* Sliding-window attention (the "swa" layer forward of the ds4.c study
   * notes, Part 4, whose listing names the variant but states no window
   * semantics): 0 = full causal attention; W > 0 = the query in slot p
   * attends slots [max(0, p - W + 1), p], the last W slots including its
   * own.  Pinned: W >= L + T equals full attention bit for bit; W = 1 gives
   * each row the output of a lone token; slots outside the window are never
   * read; a band-masked brute-force restatement agrees. */
  int64_t window;
  /* use_yarn != 0: RoPE of q and k is orc_rope_yarn with `yarn`. */
  int64_t use_yarn;
  orc_yarn yarn;
} orc_config;

/* Host pointers to fp16 bit patterns, weights [out, in] row-major. */
typedef struct {
  const uint16_t *ln1_g, *wq, *wk, *wv, *bq, *bk, *bv, *wo, *ln2_g, *w_gate,
      *w_up, *w_down;
} orc_weights;

/* binary16 <-> f64.  Pinned against numpy's float16 on every bit pattern. */
double orc_half_to_double(uint16_t h);
uint16_t orc_double_to_half(double v);

/* y = x / sqrt(mean(x^2) + eps) * g over n elements (g may be NULL = ones).
 * Pinned: constant vector closed form, scale invariance, output RMS. */
void orc_rmsnorm(const double* x, const double* g, int64_t n, double eps,
                 double* y);

/* In-place rotate_half RoPE of one head of width D at position pos.
 * Pinned: one-hot closed forms (pairing, sign, frequency), pos 0 identity,
 * pair-norm preservation, rot(a) then rot(b) == rot(a+b). */
void orc_rope(double* v, int64_t D, double pos, double theta);

/* The notes' ramp: 1 - clamp((i0/2 - low) / max(0.001, high - low), 0, 1)
 * (1 below the ramp: the original frequency; 0 above it: the scaled one).
 * Pinned: 1 at i0 = 2 low, 0 at i0 = 2 high, 1/2 half way, a step when
 * high = low. */
double orc_yarn_ramp(double low, double high, int64_t i0);

/* The notes' correction dimension: the frequency-pair index at which a
 * rotation of wavelength 2 pi base^(2d / n_dims) turns n_rot times over the
 * original context, n_dims ln(n_ctx_orig / (2 pi n_rot)) / (2 ln base).
 * Pinned by that defining property (inverse check). */
double orc_yarn_corr_dim(int64_t n_dims, int64_t n_ctx_orig, double n_rot, double base);

/* In-place rotate_half RoPE with YaRN frequencies and magnitude (readings
 * above).  Pinned: equals orc_rope when ext_factor = 0, freq_scale = 1,
 * attn_factor = 1; equals orc_rope at pos * freq_scale when ext_factor = 0
 * (position interpolation); every pair below the ramp turns as orc_rope and
 * every pair above it as the interpolated rotation, both scaled by m; a pair
 * half way up the ramp turns by the mean of the two angles. */
void orc_rope_yarn(double* v, int64_t D, double pos, double theta, const orc_yarn* y);

/* y[o] = sum_i W[o][i] * x[i] (+ b[o] when b != NULL); W fp16 [n_out, n_in].
 * Pinned: one-hot input selects a weight column; zero weights give the bias. */
void orc_linear(const uint16_t* W, const uint16_t* b, const double* x,
                int64_t n_out, int64_t n_in, double* y);

/* silu(z) = z / (1 + exp(-z)).  Pinned: silu(0)=0, limits, odd-part identity. */
double orc_silu(double z);

/* One query head against n_keys cache rows (row stride `stride` elements):
 * o = sum_j softmax_j(q . K_j * scale) V_j, with the maximum subtracted.
 * Pinned: one key -> V, identical keys -> mean of V, two-key closed form,
 * brute-force dense masked softmax on small cases. */
void orc_attend(const double* q, const uint16_t* K, const uint16_t* V,
                int64_t n_keys, int64_t D, int64_t stride, double scale,
                double* o);

/* The whole block for T new tokens on top of L history slots.
 *   x        fp16 [T, hidden]
 *   pos      int64 [T] position_ids (drive RoPE only)
 *   k_cache, v_cache  fp16 [n_kv_heads, max_ctx, head_dim], slots [0, L)
 *            read, slots [L, L+T) written, others untouched
 *   k_new, v_new      fp16 [T, n_kv_heads, head_dim] (may be NULL)
 *   rows     NULL: every row, out is [T, hidden]; else n_rows row indices,
 *            out is [n_rows, hidden] (K/V are still produced for all rows)
 * Returns 0, or -1 on a bad argument (T <= 0, L < 0, L + T > max_ctx,
 * n_heads % n_kv_heads != 0, odd head_dim, row index out of range).
 * prefill is L = 0, prefill_kv is L > 0, decode is T = 1. */
int orc_block_forward(const orc_config* cfg, const orc_weights* w,
                      const uint16_t* x, const int64_t* pos, int64_t T,
                      int64_t L, uint16_t* k_cache, uint16_t* v_cache,
                      uint16_t* k_new, uint16_t* v_new, const int64_t* rows,
                      int64_t n_rows, uint16_t* out);

/* ---- weight-only quantized projections --------------------------------------
 * The MLIR-compilation page names W4A16 and INT8 (symmetric / asymmetric)
 * weight quantization, with scales and zero points, and GPTQ / AWQ formats
 * (§2.2 on the TpuOp dialect, §3.2 on lowering TopOp to TpuOp).  It fixes no
 * layout; the readings followed here (also in the design notes):
 *   INT8  symmetric, one fp16 scale per output row:  w[o][i] = s[o] * q[o][i],
 *         q int8 in [-127, 127]
 *   int4  asymmetric, groups of `group` consecutive inputs per output row:
 *         w[o][i] = s[o][g] * (q[o][i] - z[o][g]), g = i / group, q and z in
 *         [0, 15]; two codes per byte along i, the even i in the low nibble;
 *         z one per byte
 * Activations stay fp16 (A16); the block is then the same with these f64
 * weights (orc_block_forward_f64w). */

/* w = dequantized INT8 weights, f64 [n_out, n_in].
 * Pinned: hand-computed rows (sign, row scale). */
void orc_dequant_i8(const int8_t* q, const uint16_t* scale, int64_t n_out, int64_t n_in,
                    double* w);

/* w = dequantized int4 weights, f64 [n_out, n_in]; packed uint8
 * [n_out, n_in/2], scale fp16 and zero uint8 [n_out, n_in/group].  Returns -1
 * (nothing written) unless n_in is even and a multiple of group > 0.
 * Pinned: nibble order, group boundaries and zero points by hand-computed
 * rows. */
int orc_dequant_u4(const uint8_t* packed, const uint16_t* scale, const uint8_t* zero,
                   int64_t n_out, int64_t n_in, int64_t group, double* w);

/* f64 values of the seven matrices, [out, in] row-major like orc_weights. */
typedef struct {
  const double *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down;
} orc_weights_f64;

/* orc_block_forward with the matrices taken from `m` (f64 values) and the
 * gains and biases from `w` (its matrix pointers are ignored).  Returns -1 if
 * a matrix of `m` is NULL, else as orc_block_forward.
 * Pinned: with matrices that fp16 holds exactly it equals orc_block_forward
 * on their fp16 bits, bit for bit (the same arithmetic in the same order). */
int orc_block_forward_f64w(const orc_config* cfg, const orc_weights* w,
                           const orc_weights_f64* m, const uint16_t* x, const int64_t* pos,
                           int64_t T, int64_t L, uint16_t* k_cache, uint16_t* v_cache,
                           uint16_t* k_new, uint16_t* v_new, const int64_t* rows,
                           int64_t n_rows, uint16_t* out);

/* ---- around the block stack (embedding in, logits and token out) ----------
 * Inference flow of the MLIR-compilation page (§2.3 "LLM inference
 * overview"): input tokens -> word embedding -> the stack of blocks -> LM
 * head -> logits -> a sampling step picks the next token.  The buddy-mlir
 * DeepSeek-R1 page (§6.4.4 and §6.4.6) samples greedily: the index of the
 * largest logit of the last valid position, vocabulary 151936.
 * Readings: the LM head is preceded by a final RMSNorm with gain g (the
 * Qwen2 convention; the pages do not print it), no bias; logits in f64 here;
 * ties go to the lowest index.  */

/* x[t, :] = E[ids[t], :] for t < T, fp16 bits copied.  E fp16 [vocab, H].
 * Returns -1 (and writes nothing) if an id is outside [0, vocab).
 * Pinned against array indexing of the same table. */
int orc_embed(const uint16_t* E, int64_t vocab, int64_t H, const int64_t* ids,
              int64_t T, uint16_t* x);

/* For each row t < T of x (fp16 [T, H]): y = RMSNorm(x[t]) * g (eps),
 * logits[t][v] = sum_i W[v][i] * y[i] for v < vocab (W fp16 [vocab, H]),
 * token[t] = the lowest v with the largest logit.  logits may be NULL.
 * Pinned: rows of W that are multiples of one vector (closed form), row
 * permutations, RMSNorm scale invariance, equal rows (lowest index). */
int orc_lm_head(const uint16_t* x, int64_t T, int64_t H, const uint16_t* g,
                double eps, const uint16_t* W, int64_t vocab, double* logits,
                int64_t* token);

#ifdef __cplusplus
}
#endif
#endif
