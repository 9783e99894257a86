/*
 * fp64 CPU oracle of the MoE expert layer: router, permutation, per-expert
 * SwiGLU FFN, gate-weighted combine, and the analytic backward.
 *
 * TEST INFRASTRUCTURE.  Plain, slow and meant to be checked by eye against
 * the pages; it shares no code with the CUDA path.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it.
 *
 * Parity pins (each test in tests/test_oracle_pins.py):
 *   router    brute-force sort-based top-k on numpy softmax; duplicate-column
 *             exact ties; renormalised weights sum to 1; k == E gives w == p;
 *             the renormalised weights equal a softmax over the chosen logits
 *   permute   counts sum to T*k; offsets are their exclusive scan; row_map is
 *             a permutation and src_row its inverse on tokens; stability by
 *             brute force; permute -> unpermute round trip is the identity
 *   forward   the permuted form equals the brute-force dense form; identical
 *             experts reduce the layer to one dense SwiGLU FFN (numpy); a
 *             hand-computed H = I = 1 case (tests/golden); the shared expert
 *             alone equals a dense SwiGLU FFN
 *   backward  central finite differences of the forward; the router-logit
 *             gradient of each token sums to zero
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Threads the parallel loops below run on (OpenMP's current maximum). */
int oracle_threads(void) { return omp_get_max_threads(); }

static inline double bf16_bits_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ------------------------------------------------------ permutation ([P2]) */

/* Group the T*k (token, slot) assignments by expert ("Awesome-ML-SYS-Tutorial"
 * MoE/EP guide, "Expert Parallelism": per-expert token counts, then permute
 * so that each expert's tokens are contiguous; "InternVL3.5 接入 pure FSDP2
 * 后端开发实践" §8.3: permute before the grouped matmul).
 *   counts[e]       = #{ i : ids[i] == e },  i = t*k + j
 *   offsets[e]      = sum_{e' < e} counts[e'],  offsets[E] = T*k
 *   row_map[i]      = offsets[ids[i]] + #{ i' < i : ids[i'] == ids[i] }
 *                     (stable: an expert's rows keep increasing i)
 *   src_row[row_map[i]] = i / k   (the token each permuted row came from)
 * Returns 0, or -1 when an id is outside [0, E). */
int oracle_permute(int64_t T, int64_t k, int64_t E, const int32_t* ids, int32_t* counts,
                   int32_t* offsets, int32_t* row_map, int32_t* src_row) {
  const int64_t R = T * k;
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < R; ++i) {
    if (ids[i] < 0 || ids[i] >= E) return -1;
    counts[ids[i]] += 1;
  }
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)calloc((size_t)(E > 0 ? E : 1), sizeof(int32_t));
  for (int64_t i = 0; i < R; ++i) {
    const int32_t e = ids[i];
    const int32_t row = offsets[e] + fill[e];
    fill[e] += 1;
    row_map[i] = row;
    src_row[row] = (int32_t)(i / k);
  }
  free(fill);
  return 0;
}

/* The permuted copy of the tokens: x_perm[row] = x[src_row[row]]
 * (the "dispatch" half of permute, as rows). */
void oracle_permute_rows(int64_t R, int64_t H, const double* x, const int32_t* src_row,
                         double* x_perm) {
  for (int64_t row = 0; row < R; ++row)
    for (int64_t c = 0; c < H; ++c) x_perm[row * H + c] = x[(int64_t)src_row[row] * H + c];
}

/* Unpermute with the gate-weighted combine ("Awesome-ML-SYS-Tutorial" MoE/EP
 * guide, "Expert Parallelism": the experts' outputs summed with the gate
 * weights; "InternVL3.5 接入 pure FSDP2 后端开发实践" §8.3: unpermute):
 *   y[t] = sum_{j=0}^{k-1} w[t,j] * y_perm[row_map[t*k+j]]  (+ y_shared[t])
 * summed in increasing j. */
void oracle_unpermute_combine(int64_t T, int64_t k, int64_t H, const double* y_perm,
                              const int32_t* row_map, const double* w, const double* y_shared,
                              double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t c = 0; c < H; ++c) y[t * H + c] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      const int64_t row = row_map[t * k + j];
      for (int64_t c = 0; c < H; ++c) y[t * H + c] += w[t * k + j] * y_perm[row * H + c];
    }
    if (y_shared)
      for (int64_t c = 0; c < H; ++c) y[t * H + c] += y_shared[t * H + c];
  }
}

/* ---------------------------------------- variant 1: bf16 / fp32 input bits */
#define AT uint16_t
#define RT float
#define LA(p, i) bf16_bits_to_f64((p)[(i)])
#define LR(p, i) ((double)(p)[(i)])
#define FN(name) name##_bits
#include "moe_oracle_body.h"
#undef AT
#undef RT
#undef LA
#undef LR
#undef FN

/* ------------------------------------------------ variant 2: double inputs */
#define AT double
#define RT double
#define LA(p, i) ((p)[(i)])
#define LR(p, i) ((p)[(i)])
#define FN(name) name##_f64
#include "moe_oracle_body.h"
#undef AT
#undef RT
#undef LA
#undef LR
#undef FN
