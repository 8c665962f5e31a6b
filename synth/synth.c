/*
 * Seeded synthetic inputs for the chunked TTT scan: counter-based normal and
 * uniform draws, row L2 normalisation and exact rounding to bf16 / fp32.
 *
 * This file holds none of the scan's arithmetic. It is shared by the tests and
 * the benchmark, which hand the same arrays to the CUDA library and to the fp64
 * oracle; neither of those links it.
 *
 * Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the 64-bit finaliser as published by Vigna)
 * used in counter mode, so that any element of a tensor can be drawn on its own:
 *   key(seed, stream) = mix(seed * G + mix(stream + C))
 *   x(key, n)         = mix(key + (n + 1) * G),   G = 0x9E3779B97F4A7C15
 * Uniform u in (0, 1]: ((x >> 11) + 1) * 2^-53.
 * Normal: Box and Muller (1958). Element m uses the pair p = m / 2 with
 * u1 = u(x(2p)), u2 = u(x(2p + 1)); r = sqrt(-2 ln u1); even m takes
 * r cos(2 pi u2), odd m takes r sin(2 pi u2).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return sm64_mix(seed * SM64_GAMMA + sm64_mix(stream + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t sm64_at(uint64_t key, uint64_t n) { return sm64_mix(key + (n + 1) * SM64_GAMMA); }

static inline double u01(uint64_t x) { return (double)((x >> 11) + 1) * 0x1.0p-53; }

void synth_uniform(uint64_t seed, uint64_t stream, uint64_t first, int64_t count, double* out) {
  const uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) out[i] = u01(sm64_at(key, first + (uint64_t)i));
}

void synth_normal(uint64_t seed, uint64_t stream, uint64_t first, int64_t count, double* out) {
  const uint64_t key = stream_key(seed, stream);
  const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    const uint64_t m = first + (uint64_t)i;
    const uint64_t p = m >> 1;
    const double r = sqrt(-2.0 * log(u01(sm64_at(key, 2 * p))));
    const double a = two_pi * u01(sm64_at(key, 2 * p + 1));
    out[i] = (m & 1) ? r * sin(a) : r * cos(a);
  }
}

/* Divide each row of length d by its Euclidean norm (rows of norm 0 are kept). */
void synth_normalize_rows(double* x, int64_t rows, int64_t d) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double* row = x + r * d;
    double s = 0.0;
    for (int64_t i = 0; i < d; ++i) s += row[i] * row[i];
    if (s > 0.0) {
      const double inv = 1.0 / sqrt(s);
      for (int64_t i = 0; i < d; ++i) row[i] *= inv;
    }
  }
}

/* Round to nearest bf16, ties to even, directly from fp64 (no double rounding
 * through fp32). bits[i] is the bf16 bit pattern, back[i] (if back is not
 * NULL) its exact value. */
void synth_round_bf16(const double* x, int64_t n, uint16_t* bits, double* back) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const double v = x[i];
    double r;
    if (v == 0.0 || !isfinite(v)) {
      r = v;
    } else {
      int e;
      (void)frexp(v, &e);           /* v = m * 2^e, 0.5 <= |m| < 1 */
      int s = e - 8;                /* 8 significant bits */
      if (s < -133) s = -133;       /* bf16 subnormal spacing 2^-133 */
      r = ldexp(nearbyint(ldexp(v, -s)), s);
    }
    const float f = (float)r;       /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    bits[i] = (uint16_t)(u >> 16);
    if (back) back[i] = (double)f;
  }
}

/* Round to nearest fp32, ties to even; back (optional) gets the exact value. */
void synth_round_f32(const double* x, int64_t n, float* f, double* back) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    f[i] = (float)x[i];
    if (back) back[i] = (double)f[i];
  }
}
