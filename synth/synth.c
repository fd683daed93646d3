/*
 * synth.c — host implementation of the seeded input generator (see synth.h).
 * Build with -ffp-contract=off: the normal sampler must round identically on
 * every host architecture.
 */
#include "synth.h"

#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN 0x9E3779B97F4A7C15ULL

uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_at(uint64_t key, uint64_t i) {
  return synth_mix64(key + (i + 1) * GOLDEN);
}

uint64_t synth_key(uint64_t seed, uint32_t cfg, uint32_t layer, uint32_t kind,
                   uint64_t index) {
  /* Hash chain over the fields; each step is one SplitMix64 output. */
  uint64_t k = synth_at(seed, 0x51A7u);
  k = synth_at(k ^ (uint64_t)cfg, 1);
  k = synth_at(k ^ (uint64_t)layer, 2);
  k = synth_at(k ^ (uint64_t)kind, 3);
  k = synth_at(k ^ index, 4);
  return k;
}

size_t synth_span_bytes(int H, int I) {
  size_t hi = (size_t)H * (size_t)I;
  return 3 * (hi / 2 + hi / 32);
}

int synth_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- uniform bytes -------------------------------------------------------- */

static void fill_codes(uint64_t key, size_t nbytes, uint8_t* dst) {
  /* byte j = byte (j % 8) of at(key, j / 8), little-endian */
  size_t nwords = nbytes / 8;
#pragma omp parallel for schedule(static)
  for (long long w = 0; w < (long long)nwords; ++w) {
    uint64_t v = synth_at(key, (uint64_t)w);
    for (int b = 0; b < 8; ++b) dst[(size_t)w * 8 + b] = (uint8_t)(v >> (8 * b));
  }
  size_t tail = nbytes - nwords * 8;
  if (tail) {
    uint64_t v = synth_at(key, (uint64_t)nwords);
    for (size_t b = 0; b < tail; ++b) dst[nwords * 8 + b] = (uint8_t)(v >> (8 * b));
  }
}

static void fill_scales(uint64_t key, size_t n, uint8_t* dst) {
#pragma omp parallel for schedule(static)
  for (long long j = 0; j < (long long)n; ++j) {
    uint64_t u32 = synth_at(key, (uint64_t)j) >> 32;
    dst[j] = (uint8_t)(119u + (uint32_t)((u32 * 9u) >> 32));
  }
}

void synth_expert_spans(uint64_t seed, uint32_t cfg, uint32_t layer,
                        uint32_t e0, uint32_t n_exp, int H, int I,
                        uint8_t* dst) {
  const size_t hi = (size_t)H * (size_t)I;
  const size_t qn = hi / 2, sn = hi / 32;
  const size_t span = synth_span_bytes(H, I);
  for (uint32_t n = 0; n < n_exp; ++n) {
    uint32_t e = e0 + n;
    uint8_t* p = dst + (size_t)n * span;
    for (int t = 0; t < 6; ++t) {
      uint64_t key = synth_key(seed, cfg, layer, SYNTH_KIND_EXPERT_BASE + t, e);
      if ((t & 1) == 0) { fill_codes(key, qn, p); p += qn; }
      else { fill_scales(key, sn, p); p += sn; }
    }
  }
}

void synth_words(uint64_t key, uint64_t first, uint64_t n, uint64_t* dst) {
  for (uint64_t i = 0; i < n; ++i) dst[i] = synth_at(key, first + i);
}

/* ---- normal samples ------------------------------------------------------- */

static const double LN2 = 0.69314718055994530942;
static const double TWO_PI = 6.28318530717958647692;

/* Natural log of u in (0, 1]: u = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * ln m = 2 atanh(t), t = (m - 1) / (m + 1), |t| <= 0.172, summed as a power
 * series to 16 odd terms (t^33 < 1e-25). */
static double own_log(double u) {
  int e;
  double m = frexp(u, &e);
  if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
  double t = (m - 1.0) / (m + 1.0);
  double t2 = t * t, term = t, sum = 0.0;
  for (int k = 1; k <= 31; k += 2) { sum += term / (double)k; term *= t2; }
  return 2.0 * sum + (double)e * LN2;
}

/* Taylor series on [0, pi/4]; 12 terms leave < 1e-24. */
static double own_cos_series(double x) {
  double x2 = x * x, term = 1.0, sum = 1.0;
  for (int n = 1; n <= 12; ++n) {
    term *= -x2 / (double)((2 * n - 1) * (2 * n));
    sum += term;
  }
  return sum;
}

static double own_sin_series(double x) {
  double x2 = x * x, term = x, sum = x;
  for (int n = 1; n <= 12; ++n) {
    term *= -x2 / (double)((2 * n) * (2 * n + 1));
    sum += term;
  }
  return sum;
}

/* cos(2 pi u) for u in [0, 1); the reductions are exact subtractions. */
static double own_cos_turns(double u) {
  double t = u, sign = 1.0;
  if (t > 0.5) t = 1.0 - t;
  if (t > 0.25) { t = 0.5 - t; sign = -1.0; }
  double r = (t <= 0.125) ? own_cos_series(TWO_PI * t)
                          : own_sin_series(TWO_PI * (0.25 - t));
  return sign * r;
}

static double normal_at(uint64_t key, uint64_t i) {
  uint64_t r1 = synth_at(key, 2 * i), r2 = synth_at(key, 2 * i + 1);
  double u1 = (double)((r1 >> 11) + 1) * 0x1.0p-53;  /* (0, 1] */
  double u2 = (double)(r2 >> 11) * 0x1.0p-53;        /* [0, 1) */
  return sqrt(-2.0 * own_log(u1)) * own_cos_turns(u2);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7FFFu + lsb;
  return (uint16_t)(b >> 16);
}

void synth_normal_f64(uint64_t key, uint64_t first, uint64_t n, double sigma,
                      double* dst) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i)
    dst[i] = sigma * normal_at(key, first + (uint64_t)i);
}

void synth_normal_f32(uint64_t key, uint64_t first, uint64_t n, double sigma,
                      float* dst) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i)
    dst[i] = (float)(sigma * normal_at(key, first + (uint64_t)i));
}

void synth_normal_bf16(uint64_t key, uint64_t first, uint64_t n, double sigma,
                       uint16_t* dst) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i)
    dst[i] = f32_to_bf16_rne((float)(sigma * normal_at(key, first + (uint64_t)i)));
}
