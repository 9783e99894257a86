/*
 * Seeded synthetic inputs for the MoE expert layer.
 *
 * This file draws random numbers and nothing else: it holds none of the
 * layer's arithmetic.  Both the fp64 oracle and the CUDA path read the
 * bits it writes, so they see identical inputs.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used as a counter-based
 * generator.  A stream is keyed by (seed, tensor id); element i of the
 * stream is the (i+1)-th SplitMix64 output of the stream's start state, so
 * any element can be computed on its own and the work splits over threads
 * without changing a single bit.
 *
 * Normals: Box-Muller (G. Box, M. Muller, 1958), cosine branch only; the
 * two uniforms of element i are stream outputs 2i and 2i+1.
 *
 * Build: plain C99 + OpenMP, no architecture flags, -ffp-contract=off so the
 * host arithmetic is the same on x86-64 and aarch64.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Start state of the stream (seed, tensor id). */
static inline uint64_t stream_base(uint64_t seed, uint64_t tid) {
  return mix64(mix64(seed + GOLDEN_GAMMA) ^ (tid * 0xD1B54A32D192ED03ULL));
}

/* Output number c (0-based) of the stream. */
static inline uint64_t stream_u64(uint64_t base, uint64_t c) {
  return mix64(base + (c + 1) * GOLDEN_GAMMA);
}

/* Uniform double in [0, 1) with 53 random bits. */
static inline double u01(uint64_t v) { return (double)(v >> 11) * 0x1.0p-53; }

static inline double normal_at(uint64_t base, uint64_t i) {
  double u1 = u01(stream_u64(base, 2 * i));
  double u2 = u01(stream_u64(base, 2 * i + 1));
  double r = sqrt(-2.0 * log1p(-u1)); /* 1-u1 lies in (0, 1] */
  return r * cos(6.283185307179586 * u2);
}

/* float -> bf16 bits, round to nearest even; NaN stays a quiet NaN. */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* n normals N(0, std^2), rounded to bf16 bits. */
void synth_normal_bf16(uint64_t seed, uint64_t tid, int64_t n, double std, uint16_t* out) {
  const uint64_t base = stream_base(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16((float)(std * normal_at(base, (uint64_t)i)));
}

/* n normals N(0, std^2), rounded to fp32. */
void synth_normal_f32(uint64_t seed, uint64_t tid, int64_t n, double std, float* out) {
  const uint64_t base = stream_base(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(std * normal_at(base, (uint64_t)i));
}

/* Uniform integer in [0, m) from stream output c (Lemire's multiply-shift,
 * bias below 2^-32 for m < 2^32, irrelevant for synthetic data). */
static inline int64_t uniform_below(uint64_t base, uint64_t c, int64_t m) {
  uint64_t v = stream_u64(base, c) >> 32;
  return (int64_t)((v * (uint64_t)m) >> 32);
}

/* A random permutation of 0..n-1 (Fisher-Yates, draw c = step). */
void synth_permutation(uint64_t seed, uint64_t tid, int64_t n, int32_t* out) {
  const uint64_t base = stream_base(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (int64_t i = n - 1; i > 0; --i) {
    int64_t j = uniform_below(base, (uint64_t)i, i + 1);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}

/* For each of T rows, k distinct integers from [0, E) in random order (a
 * partial Fisher-Yates per row; row t uses stream outputs t*k .. t*k+k-1).
 * Used to drive the permutation on its own, independent of any routing. */
void synth_distinct_ids(uint64_t seed, uint64_t tid, int64_t T, int k, int E, int32_t* out) {
  const uint64_t base = stream_base(seed, tid);
#pragma omp parallel
  {
    int32_t pool[4096];
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      for (int e = 0; e < E; ++e) pool[e] = e;
      for (int j = 0; j < k; ++j) {
        int64_t r = j + uniform_below(base, (uint64_t)(t * k + j), E - j);
        int32_t v = pool[r];
        pool[r] = pool[j];
        pool[j] = v;
        out[t * k + j] = v;
      }
    }
  }
}

/* For each of T rows, k integers drawn uniformly from [0, E) with repeats
 * allowed: a heavier-tailed count distribution for the permutation tests. */
void synth_uniform_ints(uint64_t seed, uint64_t tid, int64_t n, int64_t m, int32_t* out) {
  const uint64_t base = stream_base(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)uniform_below(base, (uint64_t)i, m);
}
