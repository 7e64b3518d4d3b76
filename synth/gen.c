/*
 * Seeded synthetic-input generator for the routed-MoE FFN block.
 *
 * This file holds no arithmetic of the block itself: it only draws numbers.
 * Both the CPU oracle and the CUDA path take their inputs from it.
 *
 * Every value is a pure function of (seed, tensor id, attempt, element index):
 *   key   = mix(mix(seed) ^ mix(tensor << 32 | attempt))
 *   h_i   = mix(key + (i + 1) * 0x9E3779B97F4A7C15)        (SplitMix64 stream)
 * where mix() is the SplitMix64 output function (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).
 *
 * Normal draws use Marsaglia's polar method (G. Marsaglia, T. A. Bray, "A
 * convenient method for generating normal variables", SIAM Review 6, 1964):
 * pair j takes two signed 32-bit uniforms u, v in [-1, 1) from h_j, redraws
 * them from a second stream while s = u^2 + v^2 is 0 or >= 1, and gives the
 * normals u f and v f, f = sqrt(-2 ln(s) / s); element i is member i % 2 of
 * pair i / 2.  The tails are those of a true normal (out to about 9.4 sigma
 * with 32-bit uniforms).  ln is evaluated here from its series (exact range
 * reduction, then 2 atanh) with IEEE +, -, *, / and sqrt only, so x86-64 and
 * AArch64 produce identical bits (build with -ffp-contract=off so that no
 * multiply-add is fused).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint32_t tensor, uint32_t attempt) {
  return mix64(mix64(seed + GOLDEN) ^ mix64((((uint64_t)tensor << 32) | attempt) + GOLDEN));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* ln(s) for a normal double s > 0: s = m 2^e with m in [sqrt(1/2), sqrt(2)) by exact bit
 * operations, then ln m = 2 atanh(t) = 2 (t + t^3/3 + t^5/5 + ...), t = (m - 1) / (m + 1),
 * |t| <= 0.1716; fourteen terms leave a remainder below 1e-19. */
static double ln_pos(double s) {
  uint64_t u;
  memcpy(&u, &s, 8);
  int e = (int)((u >> 52) & 0x7FFu) - 1023;
  u = (u & 0x000FFFFFFFFFFFFFULL) | 0x3FF0000000000000ULL; /* m in [1, 2) */
  double m;
  memcpy(&m, &u, 8);
  if (m > 1.4142135623730951) {
    m = m * 0.5;
    e += 1;
  }
  const double t = (m - 1.0) / (m + 1.0);
  const double t2 = t * t;
  double p = 1.0 / 27.0;
  for (int k = 12; k >= 0; --k) p = p * t2 + 1.0 / (double)(2 * k + 1);
  return (double)e * 0.6931471805599453 + 2.0 * t * p;
}

/* The two normals of pair j of the stream `key` (polar method, see the file header). */
static inline void normal_pair(uint64_t key, uint64_t j, double *z0, double *z1) {
  const uint64_t key2 = mix64(key ^ 0x5851F42D4C957F2DULL);
  uint64_t h = draw(key, j);
  for (uint64_t a = 1; a <= 256; ++a) {
    const double u = (double)((int64_t)(h >> 32) - 2147483648LL) * 4.656612873077393e-10; /* 2^-31 */
    const double v = (double)((int64_t)(h & 0xFFFFFFFFu) - 2147483648LL) * 4.656612873077393e-10;
    const double s = u * u + v * v;
    if (s > 0.0 && s < 1.0) {
      const double f = sqrt(-2.0 * ln_pos(s) / s);
      *z0 = u * f;
      *z1 = v * f;
      return;
    }
    h = draw(key2, (j << 8) + a); /* rejected (probability 1 - pi/4): a fresh pair of uniforms */
  }
  *z0 = *z1 = 0.0; /* 256 rejections in a row: never seen (probability below 1e-170) */
}

/* Element i of the standard normal stream `key`. */
static inline double unit_normal(uint64_t key, uint64_t i) {
  double z0, z1;
  normal_pair(key, i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

/* Standard normals of elements start .. start+n-1 of the stream `key` into z (pairs drawn once). */
static void normal_run(uint64_t key, uint64_t start, uint64_t n, double *z) {
  uint64_t i = start;
  const uint64_t end = start + n;
  if (i < end && (i & 1)) {
    z[0] = unit_normal(key, i);
    ++i;
  }
  for (; i + 1 < end; i += 2) normal_pair(key, i >> 1, &z[i - start], &z[i + 1 - start]);
  if (i < end) z[i - start] = unit_normal(key, i);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

#define RUN 2048 /* elements per parallel work item (even, so that no pair straddles two items) */

/* out[j] = float(mean + sigma * z) for element indices start .. start+n-1. */
void synth_normal_f32(uint64_t seed, uint32_t tensor, uint32_t attempt, uint64_t start,
                      uint64_t n, double mean, double sigma, float *out) {
  const uint64_t key = synth_key(seed, tensor, attempt);
  const uint64_t first = start & ~(uint64_t)(RUN - 1), items = (start + n - first + RUN - 1) / RUN;
#pragma omp parallel for schedule(static)
  for (int64_t it = 0; it < (int64_t)items; ++it) {
    double z[RUN];
    uint64_t i0 = first + (uint64_t)it * RUN, i1 = i0 + RUN;
    if (i0 < start) i0 = start;
    if (i1 > start + n) i1 = start + n;
    normal_run(key, i0, i1 - i0, z);
    for (uint64_t i = i0; i < i1; ++i) {
      double v = z[i - i0] * sigma;
      v = v + mean;
      out[i - start] = (float)v;
    }
  }
}

/* Same draw, multiplied by `gain` (applied before rounding), stored as bf16 (round to nearest even). */
void synth_normal_bf16(uint64_t seed, uint32_t tensor, uint32_t attempt, uint64_t start,
                       uint64_t n, double mean, double sigma, double gain, uint16_t *out) {
  const uint64_t key = synth_key(seed, tensor, attempt);
  const uint64_t first = start & ~(uint64_t)(RUN - 1), items = (start + n - first + RUN - 1) / RUN;
#pragma omp parallel for schedule(static)
  for (int64_t it = 0; it < (int64_t)items; ++it) {
    double z[RUN];
    uint64_t i0 = first + (uint64_t)it * RUN, i1 = i0 + RUN;
    if (i0 < start) i0 = start;
    if (i1 > start + n) i1 = start + n;
    normal_run(key, i0, i1 - i0, z);
    for (uint64_t i = i0; i < i1; ++i) {
      double v = z[i - i0] * sigma;
      v = v + mean;
      v = v * gain;
      out[i - start] = f32_to_bf16_rne((float)v);
    }
  }
}

/* Rows of a matrix whose row r is drawn with attempt attempts[r]:
 * out[r*row_len + c] = float(sigma * z(key(seed, tensor, attempts[r]), r*row_len + c)). */
void synth_normal_rows_f32(uint64_t seed, uint32_t tensor, const int32_t *attempts,
                           uint64_t row0, uint64_t rows, uint64_t row_len, double sigma,
                           float *out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < (int64_t)rows; ++r) {
    const uint64_t key = synth_key(seed, tensor, (uint32_t)attempts[r]);
    const uint64_t base = ((uint64_t)r + row0) * row_len;
    double z[RUN];
    for (uint64_t c0 = 0; c0 < row_len; c0 += RUN) {
      const uint64_t m = row_len - c0 < RUN ? row_len - c0 : RUN;
      normal_run(key, base + c0, m, z);
      for (uint64_t c = 0; c < m; ++c) out[(uint64_t)r * row_len + c0 + c] = (float)(z[c] * sigma);
    }
  }
}

/* Uniform integers in [lo, hi): lo + floor(u32 * (hi - lo) / 2^32). */
void synth_uniform_i32(uint64_t seed, uint32_t tensor, uint32_t attempt, uint64_t start,
                       uint64_t n, int64_t lo, int64_t hi, int32_t *out) {
  const uint64_t key = synth_key(seed, tensor, attempt);
  const uint64_t span = (uint64_t)(hi - lo);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)n; ++j) {
    uint64_t u = draw(key, start + (uint64_t)j) >> 32;
    out[j] = (int32_t)(lo + (int64_t)((u * span) >> 32));
  }
}

/* Each row r (row0 <= r < row0+rows) receives k distinct values drawn uniformly
 * from [0, n_values), in draw order; duplicates are redrawn from the next
 * counter.  Returns 0, or -1 when k > n_values. */
int synth_distinct_rows_i32(uint64_t seed, uint32_t tensor, uint64_t row0, uint64_t rows,
                            int32_t k, int32_t n_values, int32_t *out) {
  if (k > n_values || k <= 0 || k > 64) return -1;
  const uint64_t key = synth_key(seed, tensor, 0);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < (int64_t)rows; ++r) {
    int32_t *row = out + r * k;
    uint64_t ctr = ((uint64_t)r + row0) << 20;
    int have = 0;
    while (have < k) {
      uint64_t u = draw(key, ctr++) >> 32;
      int32_t v = (int32_t)((u * (uint64_t)n_values) >> 32);
      int dup = 0;
      for (int q = 0; q < have; ++q) dup |= (row[q] == v);
      if (!dup) row[have++] = v;
    }
  }
  return 0;
}

/* Fisher-Yates permutation of 0..n-1. */
void synth_permutation(uint64_t seed, uint32_t tensor, int32_t n, int32_t *out) {
  const uint64_t key = synth_key(seed, tensor, 0);
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    uint64_t u = draw(key, (uint64_t)i) >> 32;
    int32_t j = (int32_t)((u * (uint64_t)(i + 1)) >> 32);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}

/* ---- MXFP8 storage of the same draws (input preparation, not the block's arithmetic) ----------
 * OCP Microscaling (MX) format, E4M3 elements: every 32 consecutive elements share one E8M0 scale
 * X = 2^(shared_exp), shared_exp = floor(log2(max |v|)) - 8 (8: the largest exponent of an E4M3
 * value), stored as shared_exp + 127; each element is v / X rounded to the nearest E4M3 value (ties
 * to even), saturating at +-448.  E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 holds the subnormals m/8 * 2^-6; no infinities. */
static uint8_t e4m3_encode(double x) {
  const uint8_t sign = x < 0 ? 0x80u : 0u;
  double a = fabs(x);
  if (!(a < 448.0)) return sign | 0x7Eu; /* saturate (also catches the rounding to 448 below) */
  if (a < 0.015625) {                    /* below 2^-6: subnormal grid of 2^-9 */
    const double q = nearbyint(a * 512.0); /* exact scaling; ties to even */
    return sign | (uint8_t)q;            /* q == 8 is 2^-6, the smallest normal (code 0x08) */
  }
  int e;
  const double f = frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): the E4M3 exponent is e - 1 */
  double mq = nearbyint((f * 2.0 - 1.0) * 8.0);
  int ex = e - 1;
  if (mq == 8.0) {
    mq = 0.0;
    ex += 1;
  }
  const int code = ((ex + 7) << 3) | (int)mq;
  return sign | (uint8_t)(code > 0x7E ? 0x7E : code);
}

static void mx_block(const float *v, uint8_t *q, uint8_t *s) {
  double amax = 0.0;
  for (int k = 0; k < 32; ++k) amax = fmax(amax, fabs((double)v[k]));
  int shared = 0;
  if (amax > 0.0) {
    int e;
    (void)frexp(amax, &e);
    shared = (e - 1) - 8;
    if (shared < -127) shared = -127;
    if (shared > 127) shared = 127;
  }
  *s = (uint8_t)(shared + 127);
  const double inv = ldexp(1.0, -shared);
  for (int k = 0; k < 32; ++k) q[k] = e4m3_encode((double)v[k] * inv);
}

/* MXFP8 of n given values (n a multiple of 32): q[n] E4M3 codes, s[n/32] E8M0 scales. */
void synth_quantize_mxfp8(const float *v, uint64_t n, uint8_t *q, uint8_t *s) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)(n / 32); ++b) mx_block(v + 32 * b, q + 32 * b, s + b);
}

/* MXFP8 of the draws float(sigma * z) of elements start .. start+n-1 (start and n multiples of 32):
 * the same numbers synth_normal_bf16 rounds to bf16 (gain 1). */
void synth_normal_mxfp8(uint64_t seed, uint32_t tensor, uint64_t start, uint64_t n, double sigma, uint8_t *q,
                        uint8_t *s) {
  const uint64_t key = synth_key(seed, tensor, 0);
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)(n / 32); ++b) {
    float v[32];
    double z[32];
    normal_run(key, start + (uint64_t)(32 * b), 32, z);
    for (int k = 0; k < 32; ++k) {
      double x = z[k] * sigma;
      x = x + 0.0;
      v[k] = (float)x;
    }
    mx_block(v, q + 32 * b, s + b);
  }
}
