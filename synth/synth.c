/*
 * Seeded synthetic inputs for the decoder-block tests and benchmark.
 *
 * This file draws numbers and nothing else: it holds none of the block's
 * arithmetic.  Both the CPU oracle and the GPU harness take their inputs from
 * here, so the two sides see identical fp16 bit patterns.
 *
 * Generator (counter-based, so any element can be drawn independently and the
 * work can be split across threads):
 *   key      = splitmix64_mix(seed * 0x9E3779B97F4A7C15 + stream)
 *   draw(c)  = splitmix64_mix(key + (c + 1) * 0x9E3779B97F4A7C15)
 *   element i of a stream uses counters 2i and 2i+1:
 *     u1 = ((draw(2i)   >> 11) + 1) * 2^-53        in (0, 1]
 *     u2 =  (draw(2i+1) >> 11)      * 2^-53        in [0, 1)
 *     z  = sqrt(-2 ln u1) * cos(2 pi u2)           (Box-Muller, cosine branch)
 *     value = mean + std * z, rounded to IEEE binary16, nearest-even.
 * splitmix64_mix is the output function of Steele, Lea and Flood's
 * SplitMix64 ("Fast splittable pseudorandom number generators", OOPSLA 2014).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const uint64_t GOLDEN = 0x9E3779B97F4A7C15ULL;

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Round a double to the nearest binary16 value (ties to even) and return its
 * bit pattern.  Infinities and NaN pass through; overflow gives infinity. */
static uint16_t to_half_bits(double v) {
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (isnan(v)) return (uint16_t)(sign | 0x7E00u);
  if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1) */
  int e = ex - 1;                /* floor(log2 a) */
  if (e < -14) e = -14;          /* subnormal range shares the 2^-24 quantum */
  double quantum = ldexp(1.0, e - 10);
  double r = rint(a / quantum) * quantum;   /* default rounding: nearest-even */
  if (r >= 65520.0) return (uint16_t)(sign | 0x7C00u);
  if (r < ldexp(1.0, -14)) {     /* subnormal (or zero after rounding) */
    return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
  }
  frexp(r, &ex);
  int be = ex - 1 + 15;          /* biased exponent */
  double frac = r / ldexp(1.0, ex - 1) - 1.0;  /* in [0, 1), exact */
  uint16_t m = (uint16_t)(frac * 1024.0);
  return (uint16_t)(sign | (uint16_t)(be << 10) | m);
}

/* One standard-normal draw for element `i` of the stream keyed by `key`. */
static double normal_at(uint64_t key, uint64_t i) {
  uint64_t d1 = mix64(key + (2 * i + 1) * GOLDEN);
  uint64_t d2 = mix64(key + (2 * i + 2) * GOLDEN);
  double u1 = (double)((d1 >> 11) + 1) * 0x1.0p-53;
  double u2 = (double)(d2 >> 11) * 0x1.0p-53;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * GOLDEN + stream);
}

/* out[j] = fp16(mean + std * z(first + j)), j in [0, count). */
void synth_normal_f16(uint64_t seed, uint64_t stream, uint64_t first,
                      uint64_t count, double mean, double std, uint16_t* out) {
  uint64_t key = synth_stream_key(seed, stream);
  for (uint64_t j = 0; j < count; ++j)
    out[j] = to_half_bits(mean + std * normal_at(key, first + j));
}

/* Same draws in double precision (used to check the generator itself). */
void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t first,
                      uint64_t count, double* out) {
  uint64_t key = synth_stream_key(seed, stream);
  for (uint64_t j = 0; j < count; ++j) out[j] = normal_at(key, first + j);
}

/* Exposes the rounding step alone so that it can be checked against an
 * independent fp16 conversion. */
void synth_round_f16(const double* in, uint64_t count, uint16_t* out) {
  for (uint64_t j = 0; j < count; ++j) out[j] = to_half_bits(in[j]);
}
