/*
 * Body of the fp64 oracle, included twice by moe_oracle.c:
 *   - "bits": x, gate_up, down, dY and the shared expert as bf16 bits,
 *             W_r and bias as fp32  (the synthetic workloads, read exactly);
 *   - "f64":  every input as double (finite-difference pins perturb inputs).
 * The including file defines
 *   AT       storage type of x / gate_up / down / dY / shared weights
 *   RT       storage type of W_r and bias
 *   LA(p,i)  element i of an AT array as double (exact)
 *   LR(p,i)  element i of an RT array as double (exact)
 *   FN(name) name with the variant suffix.
 *
 * TEST INFRASTRUCTURE: only tests, the smoke check and the benchmark's CPU
 * baseline call this code; the product path never does.
 *
 * Sources (page titles and sections):
 *   [P4a] "InternVL3.5 接入 pure FSDP2 后端开发实践" (MindSpeed-MM issue 625)
 *         §2 (fused expert layout gate_up_proj [E*H, 2I], down_proj [E*I, H])
 *         §8.2 (router: gate -> FP32 softmax -> top-k -> weight renormalise)
 *         §8.3 (experts: permute -> grouped_matmul -> SwiGLU -> grouped_matmul
 *               -> unpermute; weights viewed as 3-D per-expert matrices)
 *   [P2]  Awesome-ML-SYS-Tutorial MoE/EP guide (gsyq.cn), "Expert Parallelism":
 *         plain MoE forward (gate scores, expert choice, dispatch, expert
 *         compute, combine as the gate-weighted sum), shared experts that are
 *         always active, per-expert token counts and permute by expert.
 */

/* ---------------------------------------------------------------- router */

/* Router for every token ([P4a] §8.2, [P2] "gate" step).
 *   z[t,e]  = sum_h x[t,h] * W_r[h,e] + bias[e]           (fp64)
 *   p[t,:]  = softmax(z[t,:])
 *   ids[t,:]= the k experts of largest p, largest first; equal p -> lower
 *             expert index first
 *   w[t,j]  = p[t,ids[t,j]] / sum_i p[t,ids[t,i]]        (renormalised)
 * kgap[t]  = z of the k-th chosen expert minus the largest z left out
 *            (+inf when k == E): how close the selection was to a tie.
 * ordgap[t]= smallest z difference between consecutive chosen experts
 *            (+inf when k == 1): how close the order was to a tie.
 * logits (nullable) receives z, probs (nullable) receives p. */
void FN(oracle_route)(int64_t T, int64_t H, int64_t E, int64_t k, const AT* x, const RT* w_r,
                      const RT* bias, double* logits, double* probs, int32_t* ids, double* w,
                      double* kgap, double* ordgap) {
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * E);
    double* p = (double*)malloc(sizeof(double) * E);
    char* taken = (char*)malloc(E);
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
      /* z[e] accumulates over h in increasing order (loop nest h-outer so
       * that W_r is read along its rows) */
      for (int64_t e = 0; e < E; ++e) z[e] = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        const double xh = LA(x, t * H + h);
        for (int64_t e = 0; e < E; ++e) z[e] += xh * LR(w_r, h * E + e);
      }
      if (bias)
        for (int64_t e = 0; e < E; ++e) z[e] += LR(bias, e);
      double m = z[0];
      for (int64_t e = 1; e < E; ++e)
        if (z[e] > m) m = z[e];
      double s = 0.0;
      for (int64_t e = 0; e < E; ++e) {
        p[e] = exp(z[e] - m);
        s += p[e];
      }
      for (int64_t e = 0; e < E; ++e) p[e] /= s;
      if (logits)
        for (int64_t e = 0; e < E; ++e) logits[t * E + e] = z[e];
      if (probs)
        for (int64_t e = 0; e < E; ++e) probs[t * E + e] = p[e];

      /* top-k by repeated selection: scan experts in increasing index and keep
       * the first maximum, so equal probabilities go to the lower index. */
      memset(taken, 0, E);
      double psum = 0.0;
      for (int64_t j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e)
          if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
        taken[best] = 1;
        ids[t * k + j] = (int32_t)best;
        psum += p[best];
      }
      for (int64_t j = 0; j < k; ++j) w[t * k + j] = p[ids[t * k + j]] / psum;

      if (kgap) {
        double zk = z[ids[t * k + k - 1]];
        double zout = -INFINITY;
        for (int64_t e = 0; e < E; ++e)
          if (!taken[e] && z[e] > zout) zout = z[e];
        kgap[t] = (k == E) ? INFINITY : zk - zout;
      }
      if (ordgap) {
        double g = INFINITY;
        for (int64_t j = 0; j + 1 < k; ++j) {
          double d = z[ids[t * k + j]] - z[ids[t * k + j + 1]];
          if (d < g) g = d;
        }
        ordgap[t] = g;
      }
    }
    free(z);
    free(p);
    free(taken);
  }
}

/* ------------------------------------------------------- expert FFN (one row) */

static inline double FN(silu)(double v) { return v / (1.0 + exp(-v)); }

/* One token through one SwiGLU expert ([P4a] §2 and §8.3).  The expert's
 * gate_up block is the H x 2I matrix whose columns 0..I-1 are the gate (SiLU)
 * branch and I..2I-1 the up branch; its down block is I x H.
 *   g = a . Wg,  u = a . Wu,  hv = silu(g) * u,  f = hv . Wd
 * g_out/u_out/h_out/f_out are nullable except f_out. */
static void FN(ffn_row)(int64_t H, int64_t I, const AT* a, const AT* gu_e, const AT* dn_e,
                        double* g_out, double* u_out, double* h_out, double* f_out) {
  /* Every sum runs over its contraction index in increasing order; the loop
   * nests put that index outside so the weights are read along their rows. */
  double* g = (double*)calloc((size_t)I, sizeof(double));
  double* u = (double*)calloc((size_t)I, sizeof(double));
  double* hv = (double*)malloc(sizeof(double) * I);
  for (int64_t h = 0; h < H; ++h) {
    const double ah = LA(a, h);
    const AT* row = gu_e + h * 2 * I;
    for (int64_t i = 0; i < I; ++i) {
      g[i] += ah * LA(row, i);
      u[i] += ah * LA(row, I + i);
    }
  }
  for (int64_t i = 0; i < I; ++i) {
    hv[i] = FN(silu)(g[i]) * u[i];
    if (g_out) g_out[i] = g[i];
    if (u_out) u_out[i] = u[i];
    if (h_out) h_out[i] = hv[i];
  }
  for (int64_t c = 0; c < H; ++c) f_out[c] = 0.0;
  for (int64_t i = 0; i < I; ++i) {
    const AT* row = dn_e + i * H;
    for (int64_t c = 0; c < H; ++c) f_out[c] += hv[i] * LA(row, c);
  }
  free(g);
  free(u);
  free(hv);
}

/* A dense SwiGLU FFN on every row of a [T, H] input (the shared expert, which
 * every token passes through with weight 1; [P2] "shared experts").
 * gu: [H, 2I], dn: [I, H]; y: [T, H]. */
void FN(oracle_dense_ffn)(int64_t T, int64_t H, int64_t I, const AT* x, const AT* gu, const AT* dn,
                          double* y) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) FN(ffn_row)(H, I, x + t * H, gu, dn, NULL, NULL, NULL, y + t * H);
}

/* ------------------------------------------------ forward, permuted form */

/* The layer as the pages lay it out ([P4a] §8.3): rows grouped by expert by
 * the permutation (offsets, src_row), each expert's FFN run on its rows, then
 * unpermute with the gate-weighted combine ([P2] "combine"):
 *   y[t] = sum_j w[t,j] * y_perm[row_map[t*k+j]]   (+ shared expert of x[t])
 * Optional outputs: gu_perm [R, 2I] (pre-activations g | u), h_perm [R, I],
 * y_perm [R, H], y_shared [T, H]. */
void FN(oracle_forward_permuted)(int64_t T, int64_t H, int64_t E, int64_t k, int64_t I, const AT* x,
                                 const AT* gate_up, const AT* down, const double* w,
                                 const int32_t* offsets, const int32_t* row_map,
                                 const int32_t* src_row, int64_t I_s, const AT* sh_gu,
                                 const AT* sh_dn, double* gu_perm, double* h_perm, double* y_perm,
                                 double* y_shared, double* y) {
  const int64_t R = T * k;
  double* yp = y_perm ? y_perm : (double*)malloc(sizeof(double) * R * H);
  for (int64_t e = 0; e < E; ++e) {
    const AT* gu_e = gate_up + e * H * 2 * I;
    const AT* dn_e = down + e * I * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t row = offsets[e]; row < offsets[e + 1]; ++row) {
      const int64_t t = src_row[row];
      FN(ffn_row)(H, I, x + t * H, gu_e, dn_e, gu_perm ? gu_perm + row * 2 * I : NULL,
                  gu_perm ? gu_perm + row * 2 * I + I : NULL, h_perm ? h_perm + row * I : NULL,
                  yp + row * H);
    }
  }
  double* ysh = NULL;
  if (I_s > 0) {
    ysh = y_shared ? y_shared : (double*)malloc(sizeof(double) * T * H);
    FN(oracle_dense_ffn)(T, H, I_s, x, sh_gu, sh_dn, ysh);
  }
  oracle_unpermute_combine(T, k, H, yp, row_map, w, ysh, y);
  if (ysh && !y_shared) free(ysh);
  if (!y_perm) free(yp);
}

/* ------------------------------------------- forward, brute-force dense form */

/* Every expert on every token, then masked by the routing: an independent
 * path to the same y ([P2] plain MoE forward, without any grouping):
 *   y[t] = sum_e m[t,e] * FFN_e(x[t])  (+ shared),  m[t,e] = w[t,j] if
 *   ids[t,j] == e, else 0. */
void FN(oracle_forward_dense)(int64_t T, int64_t H, int64_t E, int64_t k, int64_t I, const AT* x,
                              const AT* gate_up, const AT* down, const int32_t* ids,
                              const double* w, int64_t I_s, const AT* sh_gu, const AT* sh_dn,
                              double* y) {
#pragma omp parallel
  {
    double* f = (double*)malloc(sizeof(double) * H);
    double* m = (double*)malloc(sizeof(double) * E);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      for (int64_t e = 0; e < E; ++e) m[e] = 0.0;
      for (int64_t j = 0; j < k; ++j) m[ids[t * k + j]] = w[t * k + j];
      for (int64_t c = 0; c < H; ++c) y[t * H + c] = 0.0;
      for (int64_t e = 0; e < E; ++e) {
        FN(ffn_row)(H, I, x + t * H, gate_up + e * H * 2 * I, down + e * I * H, NULL, NULL, NULL, f);
        for (int64_t c = 0; c < H; ++c) y[t * H + c] += m[e] * f[c];
      }
      if (I_s > 0) {
        FN(ffn_row)(H, I_s, x + t * H, sh_gu, sh_dn, NULL, NULL, NULL, f);
        for (int64_t c = 0; c < H; ++c) y[t * H + c] += f[c];
      }
    }
    free(f);
    free(m);
  }
}

/* ------------------------------------------ forward, per-token definition */

/* The definition on a list of tokens only (large workloads are checked on a
 * seeded token sample):  y = sum_j w[t,j] * FFN_{ids[t,j]}(x[t]) (+ shared).
 * f_out (nullable) receives the k expert outputs [ntok, k, H]. */
void FN(oracle_forward_tokens)(int64_t ntok, const int64_t* tok, int64_t H, int64_t E, int64_t k,
                               int64_t I, const AT* x, const AT* gate_up, const AT* down,
                               const int32_t* ids, const double* w, int64_t I_s, const AT* sh_gu,
                               const AT* sh_dn, double* y, double* f_out) {
  (void)E;
#pragma omp parallel
  {
    double* f = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
    for (int64_t n = 0; n < ntok; ++n) {
      const int64_t t = tok[n];
      for (int64_t c = 0; c < H; ++c) y[n * H + c] = 0.0;
      for (int64_t j = 0; j < k; ++j) {
        const int64_t e = ids[t * k + j];
        FN(ffn_row)(H, I, x + t * H, gate_up + e * H * 2 * I, down + e * I * H, NULL, NULL, NULL, f);
        for (int64_t c = 0; c < H; ++c) y[n * H + c] += w[t * k + j] * f[c];
        if (f_out)
          for (int64_t c = 0; c < H; ++c) f_out[(n * k + j) * H + c] = f[c];
      }
      if (I_s > 0) {
        FN(ffn_row)(H, I_s, x + t * H, sh_gu, sh_dn, NULL, NULL, NULL, f);
        for (int64_t c = 0; c < H; ++c) y[n * H + c] += f[c];
      }
    }
    free(f);
  }
}

/* ------------------------------------------------------------- backward */

/* Backward of one token (the analytic gradient of the layer with the chosen
 * expert set held fixed; the loss is L = sum_t <dY[t], y[t]>):
 *   f_j       = FFN_{e_j}(x),  dw_j = <dY, f_j>
 *   dz_{e_j}  = w_j * (dw_j - sum_i w_i dw_i),  dz_e = 0 for unchosen e
 *               (w is the softmax restricted to the chosen logits)
 *   dhv       = w_j * (Wd_e . dY)
 *   du        = dhv * silu(g),   dg = dhv * u * silu'(g),
 *   silu'(g)  = s(g) * (1 + g * (1 - s(g))), s the logistic function
 *   dX        = sum_j (Wg_e . dg + Wu_e . du) + W_r . dz
 * dX: [H], dz: [E] (overwritten), dw: [k]. */
static void FN(backward_token)(int64_t t, int64_t H, int64_t E, int64_t k, int64_t I, const AT* x,
                               const RT* w_r, const AT* gate_up, const AT* down,
                               const int32_t* ids, const double* w, const AT* dy, double* dX,
                               double* dz, double* dw) {
  double* g = (double*)malloc(sizeof(double) * I);
  double* u = (double*)malloc(sizeof(double) * I);
  double* dg = (double*)malloc(sizeof(double) * I);
  double* du = (double*)malloc(sizeof(double) * I);
  double* f = (double*)malloc(sizeof(double) * H);
  const AT* a = x + t * H;
  const AT* d = dy + t * H;
  for (int64_t c = 0; c < H; ++c) dX[c] = 0.0;
  for (int64_t e = 0; e < E; ++e) dz[e] = 0.0;
  for (int64_t j = 0; j < k; ++j) {
    const int64_t e = ids[t * k + j];
    const AT* gu_e = gate_up + e * H * 2 * I;
    const AT* dn_e = down + e * I * H;
    FN(ffn_row)(H, I, a, gu_e, dn_e, g, u, NULL, f);
    double acc = 0.0;
    for (int64_t c = 0; c < H; ++c) acc += LA(d, c) * f[c];
    dw[j] = acc;
    const double wj = w[t * k + j];
    for (int64_t i = 0; i < I; ++i) {
      double dh = 0.0;
      for (int64_t c = 0; c < H; ++c) dh += LA(dn_e, i * H + c) * LA(d, c);
      dh *= wj;
      const double sg = 1.0 / (1.0 + exp(-g[i]));
      du[i] = dh * g[i] * sg;                                  /* dh * silu(g) */
      dg[i] = dh * u[i] * sg * (1.0 + g[i] * (1.0 - sg));      /* dh * u * silu'(g) */
    }
    for (int64_t c = 0; c < H; ++c) {
      const AT* row = gu_e + c * 2 * I;
      double s = 0.0;
      for (int64_t i = 0; i < I; ++i) s += LA(row, i) * dg[i] + LA(row, I + i) * du[i];
      dX[c] += s;
    }
  }
  double mean = 0.0;
  for (int64_t j = 0; j < k; ++j) mean += w[t * k + j] * dw[j];
  for (int64_t j = 0; j < k; ++j) dz[ids[t * k + j]] = w[t * k + j] * (dw[j] - mean);
  for (int64_t c = 0; c < H; ++c) {
    double acc = 0.0;
    for (int64_t e = 0; e < E; ++e) acc += LR(w_r, c * E + e) * dz[e];
    dX[c] += acc;
  }
  free(g);
  free(u);
  free(dg);
  free(du);
  free(f);
}

/* dX and the router-logit gradient for a list of tokens.
 * dX: [ntok, H], dlogits: [ntok, E], dw (nullable): [ntok, k]. */
void FN(oracle_backward_tokens)(int64_t ntok, const int64_t* tok, int64_t H, int64_t E, int64_t k,
                                int64_t I, const AT* x, const RT* w_r, const AT* gate_up,
                                const AT* down, const int32_t* ids, const double* w, const AT* dy,
                                double* dX, double* dlogits, double* dw) {
#pragma omp parallel
  {
    double* dwl = (double*)malloc(sizeof(double) * k);
#pragma omp for schedule(dynamic, 1)
    for (int64_t n = 0; n < ntok; ++n) {
      FN(backward_token)(tok[n], H, E, k, I, x, w_r, gate_up, down, ids, w, dy, dX + n * H,
                         dlogits + n * E, dwl);
      if (dw)
        for (int64_t j = 0; j < k; ++j) dw[n * k + j] = dwl[j];
    }
    free(dwl);
  }
}

/* Weight gradients of one expert e, summed over the rows (t, j) with
 * ids[t,j] == e taken in increasing t:
 *   d_down_e[i,c]    = sum_rows hv_i * w_j * dY[t,c]
 *   d_gate_up_e[h,i] = sum_rows x[t,h] * dg_i,  d_gate_up_e[h,I+i] = sum_rows x[t,h] * du_i
 * with hv, dg, du of the row as in the per-token backward.
 * dgu_e: [H, 2I], ddn_e: [I, H] (overwritten; zero when no token chose e). */
void FN(oracle_backward_expert)(int64_t e, int64_t T, int64_t H, int64_t k, int64_t I, const AT* x,
                                const AT* gate_up, const AT* down, const int32_t* ids,
                                const double* w, const AT* dy, double* dgu_e, double* ddn_e) {
  const AT* gu_e = gate_up + e * H * 2 * I;
  const AT* dn_e = down + e * I * H;
  int64_t M = 0;
  for (int64_t q = 0; q < T * k; ++q) M += (ids[q] == e);
  int64_t* rt = (int64_t*)malloc(sizeof(int64_t) * (M > 0 ? M : 1));  /* token of each row */
  double* rw = (double*)malloc(sizeof(double) * (M > 0 ? M : 1));     /* its gate weight */
  int64_t m = 0;
  for (int64_t q = 0; q < T * k; ++q)
    if (ids[q] == e) {
      rt[m] = q / k;
      rw[m] = w[q];
      ++m;
    }
  double* hv = (double*)malloc(sizeof(double) * (M * I > 0 ? M * I : 1));
  double* dg = (double*)malloc(sizeof(double) * (M * I > 0 ? M * I : 1));
  double* du = (double*)malloc(sizeof(double) * (M * I > 0 ? M * I : 1));
#pragma omp parallel
  {
    double* g = (double*)malloc(sizeof(double) * I);
    double* u = (double*)malloc(sizeof(double) * I);
    double* f = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < M; ++r) {
      const AT* d = dy + rt[r] * H;
      FN(ffn_row)(H, I, x + rt[r] * H, gu_e, dn_e, g, u, hv + r * I, f);
      for (int64_t i = 0; i < I; ++i) {
        double dh = 0.0;
        for (int64_t c = 0; c < H; ++c) dh += LA(dn_e, i * H + c) * LA(d, c);
        dh *= rw[r];
        const double sg = 1.0 / (1.0 + exp(-g[i]));
        du[r * I + i] = dh * g[i] * sg;
        dg[r * I + i] = dh * u[i] * sg * (1.0 + g[i] * (1.0 - sg));
      }
    }
    free(g);
    free(u);
    free(f);
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < I; ++i) {
    double* out = ddn_e + i * H;
    for (int64_t c = 0; c < H; ++c) out[c] = 0.0;
    for (int64_t r = 0; r < M; ++r) {
      const double s = hv[r * I + i] * rw[r];
      const AT* d = dy + rt[r] * H;
      for (int64_t c = 0; c < H; ++c) out[c] += s * LA(d, c);
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t h = 0; h < H; ++h) {
    double* out = dgu_e + h * 2 * I;
    for (int64_t i = 0; i < 2 * I; ++i) out[i] = 0.0;
    for (int64_t r = 0; r < M; ++r) {
      const double ah = LA(x, rt[r] * H + h);
      for (int64_t i = 0; i < I; ++i) {
        out[i] += ah * dg[r * I + i];
        out[I + i] += ah * du[r * I + i];
      }
    }
  }
  free(rt);
  free(rw);
  free(hv);
  free(dg);
  free(du);
}

/* The whole backward: dX [T,H], dlogits [T,E], dw (nullable) [T,k], and the
 * weight gradients d_gate_up [E*H, 2I], d_down [E*I, H], d_w_r [H, E]
 * (each nullable).  d_w_r[h,e] = sum_t x[t,h] * dz[t,e]. */
void FN(oracle_backward)(int64_t T, int64_t H, int64_t E, int64_t k, int64_t I, const AT* x,
                         const RT* w_r, const AT* gate_up, const AT* down, const int32_t* ids,
                         const double* w, const AT* dy, double* dX, double* dlogits, double* dw,
                         double* d_gate_up, double* d_down, double* d_w_r) {
  int64_t* tok = (int64_t*)malloc(sizeof(int64_t) * (T > 0 ? T : 1));
  for (int64_t t = 0; t < T; ++t) tok[t] = t;
  FN(oracle_backward_tokens)(T, tok, H, E, k, I, x, w_r, gate_up, down, ids, w, dy, dX, dlogits, dw);
  free(tok);
  if (d_gate_up && d_down)
    for (int64_t e = 0; e < E; ++e)
      FN(oracle_backward_expert)(e, T, H, k, I, x, gate_up, down, ids, w, dy,
                                 d_gate_up + e * H * 2 * I, d_down + e * I * H);
  if (d_w_r) {
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < H; ++h)
      for (int64_t e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int64_t t = 0; t < T; ++t) acc += LA(x, t * H + h) * dlogits[t * E + e];
        d_w_r[h * E + e] = acc;
      }
  }
}
