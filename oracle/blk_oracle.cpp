// CPU oracle for one Qwen2-style decoder block — TEST INFRASTRUCTURE ONLY.
// The contract, the readings of the source pages and the pin of every
// function are in blk_oracle.h.  Plain single-threaded f64 loops, summed in
// ascending index order; no blocking, fusion or reordering.
#include "blk_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

namespace {

// Exact binary16 -> f64 for one bit pattern.
double decode_half(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int exp = (h >> 10) & 0x1F;
  const int man = h & 0x3FF;
  double mag;
  if (exp == 0) {
    mag = std::ldexp(static_cast<double>(man), -24);  // zero or subnormal
  } else if (exp == 31) {
    mag = man ? NAN : INFINITY;
  } else {
    mag = std::ldexp(static_cast<double>(1024 + man), exp - 25);
  }
  return sign ? -mag : mag;
}

// Lookup table over all 65536 patterns, so matrix loops stay simple.
const double* half_table() {
  static const std::vector<double> table = [] {
    std::vector<double> t(65536);
    for (int i = 0; i < 65536; ++i) t[i] = decode_half(static_cast<uint16_t>(i));
    return t;
  }();
  return table.data();
}

inline double h2d(uint16_t h) { return half_table()[h]; }

// A weight matrix [n_out][n_in] row-major: fp16 bit patterns (the block's own
// weights) or f64 values (e.g. dequantized weights); val(p, k) reads element
// k of the flat array as f64.
struct MatF16 {
  const uint16_t* p;
  static double val(const uint16_t* a, int64_t k) { return h2d(a[k]); }
};
struct MatF64 {
  const double* p;
  static double val(const double* a, int64_t k) { return a[k]; }
};

// y[o] = sum_i W[o][i] * x[i] (+ b[o]), i ascending.
template <class M>
void linear(const M& W, const uint16_t* b, const double* x, int64_t n_out, int64_t n_in,
            double* y) {
  for (int64_t o = 0; o < n_out; ++o) {
    const auto* row = W.p + o * n_in;
    double acc = 0.0;
    for (int64_t i = 0; i < n_in; ++i) acc += M::val(row, i) * x[i];
    y[o] = b ? acc + h2d(b[o]) : acc;
  }
}

// f64 -> binary16, round to nearest, ties to even, on the bit pattern.
uint16_t encode_half(double v) {
  uint64_t b;
  std::memcpy(&b, &v, sizeof b);
  const uint16_t sign = static_cast<uint16_t>((b >> 63) << 15);
  const int e = static_cast<int>((b >> 52) & 0x7FF);
  const uint64_t m = b & ((1ULL << 52) - 1);
  if (e == 0x7FF) return static_cast<uint16_t>(sign | 0x7C00 | (m ? 0x200 : 0));
  if (e == 0) return sign;  // f64 subnormals are far below the fp16 range
  const int he = e - 1023 + 15;  // biased fp16 exponent if the value is normal
  if (he >= 31) return static_cast<uint16_t>(sign | 0x7C00);
  if (he <= 0) {
    // fp16 subnormal: count units of 2^-24.
    const uint64_t M = (1ULL << 52) | m;  // value = M * 2^(e - 1075)
    const int shift = 1051 - e;           // M >> shift = value / 2^-24
    if (shift > 53) return sign;
    const uint64_t q = M >> shift;
    const uint64_t rem = M & ((1ULL << shift) - 1);
    const uint64_t half = 1ULL << (shift - 1);
    const uint64_t r = q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0);
    return static_cast<uint16_t>(sign | r);  // r == 1024 encodes 2^-14 exactly
  }
  const uint64_t q = m >> 42;
  const uint64_t rem = m & ((1ULL << 42) - 1);
  const uint64_t half = 1ULL << 41;
  const uint64_t r = q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0);
  // A mantissa carry moves into the exponent field, which is the right value
  // (and reaches the infinity pattern exactly at the overflow boundary).
  return static_cast<uint16_t>(sign | ((static_cast<uint64_t>(he) << 10) + r));
}

}  // namespace

extern "C" {

double orc_half_to_double(uint16_t h) { return decode_half(h); }

uint16_t orc_double_to_half(double v) { return encode_half(v); }

void orc_rmsnorm(const double* x, const double* g, int64_t n, double eps,
                 double* y) {
  double sum_sq = 0.0;
  for (int64_t i = 0; i < n; ++i) sum_sq += x[i] * x[i];
  const double r = 1.0 / std::sqrt(sum_sq / static_cast<double>(n) + eps);
  for (int64_t i = 0; i < n; ++i) y[i] = x[i] * r * (g ? g[i] : 1.0);
}

void orc_rope(double* v, int64_t D, double pos, double theta) {
  const int64_t half = D / 2;
  for (int64_t i = 0; i < half; ++i) {
    const double inv_freq =
        std::pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(D));
    const double angle = pos * inv_freq;
    const double c = std::cos(angle), s = std::sin(angle);
    const double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

double orc_yarn_ramp(double low, double high, int64_t i0) {
  const double y = (static_cast<double>(i0 / 2) - low) / std::max(0.001, high - low);
  return 1.0 - std::min(1.0, std::max(0.0, y));
}

double orc_yarn_corr_dim(int64_t n_dims, int64_t n_ctx_orig, double n_rot, double base) {
  const double pi = 3.14159265358979323846;
  return static_cast<double>(n_dims) *
         std::log(static_cast<double>(n_ctx_orig) / (n_rot * 2.0 * pi)) / (2.0 * std::log(base));
}

void orc_rope_yarn(double* v, int64_t D, double pos, double theta, const orc_yarn* y) {
  const int64_t half = D / 2;
  const double low = orc_yarn_corr_dim(D, y->n_ctx_orig, y->beta_fast, theta);
  const double high = orc_yarn_corr_dim(D, y->n_ctx_orig, y->beta_slow, theta);
  const double m = y->ext_factor != 0.0
                       ? y->attn_factor * (1.0 + 0.1 * std::log(1.0 / y->freq_scale))
                       : y->attn_factor;
  for (int64_t i = 0; i < half; ++i) {
    const double inv_freq =
        std::pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(D));
    const double a_orig = pos * inv_freq;
    const double a_int = y->freq_scale * a_orig;
    const double r = orc_yarn_ramp(low, high, 2 * i) * y->ext_factor;
    const double angle = a_int * (1.0 - r) + a_orig * r;
    const double c = std::cos(angle) * m, s = std::sin(angle) * m;
    const double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

void orc_linear(const uint16_t* W, const uint16_t* b, const double* x,
                int64_t n_out, int64_t n_in, double* y) {
  linear(MatF16{W}, b, x, n_out, n_in, y);
}

double orc_silu(double z) { return z / (1.0 + std::exp(-z)); }

void orc_attend(const double* q, const uint16_t* K, const uint16_t* V,
                int64_t n_keys, int64_t D, int64_t stride, double scale,
                double* o) {
  std::vector<double> s(static_cast<size_t>(n_keys));
  double m = -INFINITY;
  for (int64_t j = 0; j < n_keys; ++j) {
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += q[d] * h2d(K[j * stride + d]);
    s[j] = dot * scale;
    if (s[j] > m) m = s[j];
  }
  double denom = 0.0;
  for (int64_t j = 0; j < n_keys; ++j) {
    s[j] = std::exp(s[j] - m);
    denom += s[j];
  }
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < n_keys; ++j)
    for (int64_t d = 0; d < D; ++d) o[d] += s[j] * h2d(V[j * stride + d]);
  for (int64_t d = 0; d < D; ++d) o[d] /= denom;
}

}  // extern "C"

namespace {

// RoPE of one head at position pos: plain, or YaRN when the config asks.
void rope_of(const orc_config* cfg, double* v, int64_t pos) {
  if (cfg->use_yarn)
    orc_rope_yarn(v, cfg->head_dim, static_cast<double>(pos), cfg->rope_theta, &cfg->yarn);
  else
    orc_rope(v, cfg->head_dim, static_cast<double>(pos), cfg->rope_theta);
}

// The block with its seven matrices given as views (gains and biases are
// always fp16 from `w`).
template <class M>
int block_forward(const orc_config* cfg, const orc_weights* w, const M& wq, const M& wk,
                  const M& wv, const M& wo, const M& w_gate, const M& w_up, const M& w_down,
                  const uint16_t* x, const int64_t* pos, int64_t T, int64_t L,
                  uint16_t* k_cache, uint16_t* v_cache, uint16_t* k_new, uint16_t* v_new,
                  const int64_t* rows, int64_t n_rows, uint16_t* out) {
  const int64_t H = cfg->hidden, Hq = cfg->n_heads, Hkv = cfg->n_kv_heads;
  const int64_t D = cfg->head_dim, I = cfg->intermediate, C = cfg->max_ctx;
  if (T <= 0 || L < 0 || L + T > C || Hkv <= 0 || Hq % Hkv != 0 || D % 2 != 0 ||
      cfg->window < 0)
    return -1;
  const int64_t group = Hq / Hkv;
  const bool bias = cfg->has_qkv_bias != 0;
  const double scale = 1.0 / std::sqrt(static_cast<double>(D));

  std::vector<double> ln1(H), ln2(H);
  for (int64_t i = 0; i < H; ++i) {
    ln1[i] = h2d(w->ln1_g[i]);
    ln2[i] = h2d(w->ln2_g[i]);
  }

  // Step 1, every new row: RMSNorm, K/V projections, RoPE on K, store K/V
  // rounded to fp16 in slot L + t (and in k_new / v_new).
  std::vector<double> xn(static_cast<size_t>(T * H)), xrow(H), k(Hkv * D),
      v(Hkv * D);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t i = 0; i < H; ++i) xrow[i] = h2d(x[t * H + i]);
    orc_rmsnorm(xrow.data(), ln1.data(), H, cfg->rms_eps, &xn[t * H]);
    linear(wk, bias ? w->bk : nullptr, &xn[t * H], Hkv * D, H, k.data());
    linear(wv, bias ? w->bv : nullptr, &xn[t * H], Hkv * D, H, v.data());
    for (int64_t g = 0; g < Hkv; ++g) {
      rope_of(cfg, &k[g * D], pos[t]);
      for (int64_t d = 0; d < D; ++d) {
        const uint16_t kh = encode_half(k[g * D + d]);
        const uint16_t vh = encode_half(v[g * D + d]);
        k_cache[(g * C + L + t) * D + d] = kh;
        v_cache[(g * C + L + t) * D + d] = vh;
        if (k_new) k_new[(t * Hkv + g) * D + d] = kh;
        if (v_new) v_new[(t * Hkv + g) * D + d] = vh;
      }
    }
  }

  // Step 2, each requested row: Q, RoPE on Q, attention over slots
  // [0, L + t] (or the window's part of them), o_proj + residual, RMSNorm,
  // SwiGLU MLP + residual.
  const int64_t count = rows ? n_rows : T;
  std::vector<double> q(Hq * D), attn(Hq * D), h(H), hn(H), gate(I), up(I),
      act(I), mlp(H);
  for (int64_t r = 0; r < count; ++r) {
    const int64_t t = rows ? rows[r] : r;
    if (t < 0 || t >= T) return -1;
    linear(wq, bias ? w->bq : nullptr, &xn[t * H], Hq * D, H, q.data());
    for (int64_t hq = 0; hq < Hq; ++hq) {
      rope_of(cfg, &q[hq * D], pos[t]);
      const int64_t g = hq / group;
      // slots [lo, L + t]: all of them, or the last `window` (sliding window)
      const int64_t lo =
          (cfg->window > 0 && L + t + 1 > cfg->window) ? L + t + 1 - cfg->window : 0;
      orc_attend(&q[hq * D], &k_cache[(g * C + lo) * D], &v_cache[(g * C + lo) * D],
                 L + t + 1 - lo, D, D, scale, &attn[hq * D]);
    }
    linear(wo, nullptr, attn.data(), H, Hq * D, h.data());
    for (int64_t i = 0; i < H; ++i) h[i] += h2d(x[t * H + i]);
    orc_rmsnorm(h.data(), ln2.data(), H, cfg->rms_eps, hn.data());
    linear(w_gate, nullptr, hn.data(), I, H, gate.data());
    linear(w_up, nullptr, hn.data(), I, H, up.data());
    for (int64_t j = 0; j < I; ++j) act[j] = orc_silu(gate[j]) * up[j];
    linear(w_down, nullptr, act.data(), H, I, mlp.data());
    for (int64_t i = 0; i < H; ++i) out[r * H + i] = encode_half(h[i] + mlp[i]);
  }
  return 0;
}

}  // namespace

extern "C" {

int orc_block_forward(const orc_config* cfg, const orc_weights* w,
                      const uint16_t* x, const int64_t* pos, int64_t T,
                      int64_t L, uint16_t* k_cache, uint16_t* v_cache,
                      uint16_t* k_new, uint16_t* v_new, const int64_t* rows,
                      int64_t n_rows, uint16_t* out) {
  return block_forward(cfg, w, MatF16{w->wq}, MatF16{w->wk}, MatF16{w->wv}, MatF16{w->wo},
                       MatF16{w->w_gate}, MatF16{w->w_up}, MatF16{w->w_down}, x, pos, T, L,
                       k_cache, v_cache, k_new, v_new, rows, n_rows, out);
}

int orc_block_forward_f64w(const orc_config* cfg, const orc_weights* w,
                           const orc_weights_f64* m, const uint16_t* x, const int64_t* pos,
                           int64_t T, int64_t L, uint16_t* k_cache, uint16_t* v_cache,
                           uint16_t* k_new, uint16_t* v_new, const int64_t* rows,
                           int64_t n_rows, uint16_t* out) {
  if (!m || !m->wq || !m->wk || !m->wv || !m->wo || !m->w_gate || !m->w_up || !m->w_down)
    return -1;
  return block_forward(cfg, w, MatF64{m->wq}, MatF64{m->wk}, MatF64{m->wv}, MatF64{m->wo},
                       MatF64{m->w_gate}, MatF64{m->w_up}, MatF64{m->w_down}, x, pos, T, L,
                       k_cache, v_cache, k_new, v_new, rows, n_rows, out);
}

void orc_dequant_i8(const int8_t* q, const uint16_t* scale, int64_t n_out, int64_t n_in,
                    double* w) {
  for (int64_t o = 0; o < n_out; ++o) {
    const double s = h2d(scale[o]);
    for (int64_t i = 0; i < n_in; ++i)
      w[o * n_in + i] = s * static_cast<double>(q[o * n_in + i]);
  }
}

int orc_dequant_u4(const uint8_t* packed, const uint16_t* scale, const uint8_t* zero,
                   int64_t n_out, int64_t n_in, int64_t group, double* w) {
  if (n_in <= 0 || n_in % 2 != 0 || group <= 0 || n_in % group != 0) return -1;
  const int64_t ng = n_in / group;
  for (int64_t o = 0; o < n_out; ++o)
    for (int64_t i = 0; i < n_in; ++i) {
      const uint8_t byte = packed[o * (n_in / 2) + i / 2];
      const int code = (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
      const int64_t g = o * ng + i / group;
      w[o * n_in + i] =
          h2d(scale[g]) * (static_cast<double>(code) - static_cast<double>(zero[g]));
    }
  return 0;
}

int orc_embed(const uint16_t* E, int64_t vocab, int64_t H, const int64_t* ids,
              int64_t T, uint16_t* x) {
  if (T < 0 || H <= 0 || vocab <= 0) return -1;
  for (int64_t t = 0; t < T; ++t)
    if (ids[t] < 0 || ids[t] >= vocab) return -1;
  for (int64_t t = 0; t < T; ++t)
    for (int64_t i = 0; i < H; ++i) x[t * H + i] = E[ids[t] * H + i];
  return 0;
}

int orc_lm_head(const uint16_t* x, int64_t T, int64_t H, const uint16_t* g,
                double eps, const uint16_t* W, int64_t vocab, double* logits,
                int64_t* token) {
  if (T <= 0 || H <= 0 || vocab <= 0) return -1;
  std::vector<double> row(H), gain(H), y(H), z(vocab);
  for (int64_t i = 0; i < H; ++i) gain[i] = h2d(g[i]);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t i = 0; i < H; ++i) row[i] = h2d(x[t * H + i]);
    orc_rmsnorm(row.data(), gain.data(), H, eps, y.data());
    orc_linear(W, nullptr, y.data(), vocab, H, z.data());
    int64_t best = 0;
    for (int64_t v = 1; v < vocab; ++v)
      if (z[v] > z[best]) best = v;   // strictly larger: ties keep the lower index
    token[t] = best;
    if (logits)
      for (int64_t v = 0; v < vocab; ++v) logits[t * vocab + v] = z[v];
  }
  return 0;
}

}  // extern "C"
