/*
 * oracle.c — plain fp64 CPU reference of the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY: see oracle.h for who may call it and for the
 * sources each function follows. Nothing here is blocked, fused or reordered
 * beyond what the method states; rows are computed lazily, in the order the
 * sequential accept test reaches them, as the pages' loops do.
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------ storage */

static double load_logit(const void* base, int dtype, int64_t i) {
  if (dtype == 2) return ((const double*)base)[i];
  if (dtype == 1) {
    uint32_t u = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
  }
  return (double)((const float*)base)[i];
}

static void load_row(const void* base, int dtype, int64_t row, int64_t V, double* l) {
  for (int64_t v = 0; v < V; ++v) l[v] = load_logit(base, dtype, row * V + v);
}

/* Sampling mode: a row is usable when it holds no NaN, no +inf, and at least
 * one finite value (otherwise softmax is undefined). */
static int row_ok_sampling(const double* l, int64_t V) {
  int any_finite = 0;
  for (int64_t v = 0; v < V; ++v) {
    if (isnan(l[v]) || l[v] == INFINITY) return 0;
    if (l[v] != -INFINITY) any_finite = 1;
  }
  return any_finite;
}

static int row_has_nan(const double* l, int64_t V) {
  for (int64_t v = 0; v < V; ++v)
    if (isnan(l[v])) return 1;
  return 0;
}

/* ----------------------------------------------------- distributions */

/* Temperature-scaled softmax, [P2] §3.4 / [P1] §4: z = l / T, then
 * p_v = exp(z_v - M) / sum_w exp(z_w - M) with M = max z. Returns log of the
 * normaliser (lse) and M through the pointers. */
static void softmax_T(const double* l, int64_t V, double T, double* p, double* M_out, double* lse_out) {
  double M = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    double z = l[v] / T;
    if (z > M) M = z;
  }
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double e = (l[v] == -INFINITY) ? 0.0 : exp(l[v] / T - M);
    p[v] = e;
    S += e;
  }
  for (int64_t v = 0; v < V; ++v) p[v] /= S;
  if (M_out) *M_out = M;
  if (lse_out) *lse_out = M + log(S);
}

typedef struct {
  double val;
  int64_t idx;
} val_idx;

static int by_value_desc(const void* a, const void* b) {
  const val_idx* x = (const val_idx*)a;
  const val_idx* y = (const val_idx*)b;
  if (x->val > y->val) return -1;
  if (x->val < y->val) return 1;
  return (x->idx > y->idx) - (x->idx < y->idx);
}

/* Top-p nucleus, [P2] §3.4 and §5.2: keep the tokens whose stored logit is at
 * least tau, where tau is the largest stored value whose upper set
 * {v : l_v >= tau} holds probability >= top_p; every token tied at the cut is
 * kept. Found by sorting the row in descending order and accumulating p until
 * it reaches top_p. The kept probabilities are renormalised to sum to one
 * (p'_v = p_v / P_S), the rest set to zero. Returns P_S and tau; *margin gets
 * min(top_p - mass strictly above tau, P_S - top_p). */
static void nucleus(const double* l, double* p, int64_t V, double top_p, val_idx* scratch, double* PS_out,
                    double* tau_out, double* margin) {
  for (int64_t v = 0; v < V; ++v) {
    scratch[v].val = l[v];
    scratch[v].idx = v;
  }
  qsort(scratch, (size_t)V, sizeof(val_idx), by_value_desc);
  double cum = 0.0, tau = scratch[V - 1].val;
  for (int64_t r = 0; r < V; ++r) {
    cum += p[scratch[r].idx];
    if (cum >= top_p) {
      tau = scratch[r].val;
      break;
    }
  }
  double above = 0.0, PS = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    if (l[v] > tau) above += p[v];
    if (l[v] >= tau) PS += p[v];
  }
  for (int64_t v = 0; v < V; ++v) p[v] = (l[v] >= tau) ? p[v] / PS : 0.0;
  if (PS_out) *PS_out = PS;
  if (tau_out) *tau_out = tau;
  if (margin) {
    double m = fmin(top_p - above, PS - top_p);
    if (m < *margin) *margin = m;
  }
}

/* The sampling distribution of one row: softmax at T, then top-p. */
static void row_dist(const double* l, int64_t V, double T, double top_p, double* p, val_idx* scratch,
                     double* margin) {
  softmax_T(l, V, T, p, NULL, NULL);
  if (top_p < 1.0) nucleus(l, p, V, top_p, scratch, NULL, NULL, margin);
}

/* Inverse-CDF draw from unnormalised weights w (ascending vocabulary order):
 * the smallest t with C_t = sum_{v<=t} w_v > u * Z, Z = sum_v w_v. If rounding
 * leaves u*Z at or past the last partial sum, the largest t with w_t > 0. */
static int64_t inverse_cdf(const double* w, int64_t V, double u, double* margin) {
  double Z = 0.0;
  for (int64_t v = 0; v < V; ++v) Z += w[v];
  double target = u * Z, C = 0.0;
  for (int64_t t = 0; t < V; ++t) {
    double prev = C;
    C += w[t];
    if (C > target) {
      if (margin) {
        double m = fmin(target - prev, C - target) / Z;
        if (m < *margin) *margin = m;
      }
      return t;
    }
  }
  if (margin) *margin = 0.0;
  for (int64_t t = V - 1; t >= 0; --t)
    if (w[t] > 0.0) return t;
  return V - 1;
}

/* The draw after a rejection ([P1] §2.1-2.2): from norm(max(0, p - q)); if
 * that residual is all zero, from p itself ([P1] §4 fallback). w is V doubles
 * of scratch. */
static int64_t residual_draw(const double* p, const double* q, double* w, int64_t V, double u, double* margin) {
  double Z = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    const double d = p[v] - q[v];
    w[v] = d > 0.0 ? d : 0.0;
    Z += w[v];
  }
  return inverse_cdf(Z > 0.0 ? w : p, V, u, margin);
}

/* Argmax with the lowest index among equal maxima (numeric order, so -0 and
 * +0 tie). */
static int64_t argmax_lowest(const double* l, int64_t V) {
  int64_t best = 0;
  for (int64_t v = 1; v < V; ++v)
    if (l[v] > l[best]) best = v;
  return best;
}

/* ---------------------------------------------------------- sampling */

int oracle_verify_sample(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                         const float* uniforms, int64_t B, int32_t K, int64_t V, float temperature, float top_p,
                         int32_t* out_tokens, int32_t* out_accept_len, double* out_margin) {
  if (!target || !draft_tokens || !out_tokens || !out_accept_len) return -1;
  if (B < 0 || K < 1 || V < 2 || dtype < 0 || dtype > 2) return -1;
  if (!(temperature >= 0.0f) || !(top_p > 0.0f && top_p <= 1.0f)) return -1;
  const int greedy_limit = (temperature == 0.0f);
  if (!greedy_limit && (!draft || !uniforms)) return -1;
  const double T = (double)temperature;
  const double P = (double)top_p;

  double* lt = (double*)malloc(sizeof(double) * (size_t)V);
  double* ld = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  val_idx* scratch = (val_idx*)malloc(sizeof(val_idx) * (size_t)V);
  if (!lt || !ld || !p || !q || !w || !scratch) {
    free(lt); free(ld); free(p); free(q); free(w); free(scratch);
    return -1;
  }

  for (int64_t b = 0; b < B; ++b) {
    int32_t* out = out_tokens + b * (K + 1);
    const int32_t* x = draft_tokens + b * K;
    const float* u = greedy_limit ? NULL : uniforms + b * (K + 1);
    double margin = INFINITY;
    for (int i = 0; i <= K; ++i) out[i] = -1;

    /* Input checks cover every row and token of the sequence, whichever the
     * accept test later reaches. */
    int ok = 1;
    for (int i = 0; i < K; ++i) ok &= (x[i] >= 0 && (int64_t)x[i] < V);
    if (!greedy_limit)
      for (int i = 0; i <= K; ++i) ok &= (u[i] >= 0.0f && u[i] < 1.0f);
    for (int i = 0; ok && i <= K; ++i) {
      load_row(target, dtype, b * (K + 1) + i, V, lt);
      ok = greedy_limit ? !row_has_nan(lt, V) : row_ok_sampling(lt, V);
    }
    for (int i = 0; ok && !greedy_limit && i < K; ++i) {
      load_row(draft, dtype, b * K + i, V, ld);
      ok = row_ok_sampling(ld, V);
    }
    if (!ok) {
      out_accept_len[b] = -1;
      if (out_margin) out_margin[b] = INFINITY;
      continue;
    }

    if (greedy_limit) {
      /* T -> 0: p_i is one-hot at its argmax, so x_i is accepted iff it is
       * that argmax; the residual at a rejection and the bonus are argmaxes. */
      int j = K;
      for (int i = 0; i < K; ++i) {
        load_row(target, dtype, b * (K + 1) + i, V, lt);
        int64_t a = argmax_lowest(lt, V);
        if ((int64_t)x[i] == a) {
          out[i] = x[i];
        } else {
          out[i] = (int32_t)a;
          j = i;
          break;
        }
      }
      if (j == K) {
        load_row(target, dtype, b * (K + 1) + K, V, lt);
        out[K] = (int32_t)argmax_lowest(lt, V);
      }
      out_accept_len[b] = j;
      if (out_margin) out_margin[b] = INFINITY;
      continue;
    }

    /* [P1] §2.3: test x_0, x_1, ... in order; stop at the first rejection. */
    int j = K;
    for (int i = 0; i < K; ++i) {
      load_row(target, dtype, b * (K + 1) + i, V, lt);
      load_row(draft, dtype, b * K + i, V, ld);
      row_dist(lt, V, T, P, p, scratch, &margin); /* p_i (target) */
      row_dist(ld, V, T, P, q, scratch, &margin); /* q_i (draft)  */
      const double px = p[x[i]], qx = q[x[i]];
      /* [P1] §2.1, [P2] §3.1: alpha = min(1, p(x)/q(x)). A zero q(x) with a
       * positive p(x) gives alpha = 1 (the pages' p/(q+eps)); p(x) = 0 gives
       * alpha = 0. */
      double alpha;
      if (px == 0.0)
        alpha = 0.0;
      else if (qx == 0.0)
        alpha = 1.0;
      else
        alpha = fmin(1.0, px / qx);
      double du = fabs((double)u[i] - alpha);
      if (du < margin) margin = du;
      if ((double)u[i] < alpha) { /* [P2] §3.1: r < alpha accepts */
        out[i] = x[i];
        continue;
      }
      /* Rejected at i: draw from norm(max(0, p - q)) ([P1] §2.1-2.2); if that
       * residual is all zero, draw from p instead ([P1] §4). */
      out[i] = (int32_t)residual_draw(p, q, w, V, (double)u[K], &margin);
      j = i;
      break;
    }
    if (j == K) {
      /* All K accepted: the bonus token from the target's distribution at
       * position K ([P1] §2.3, [P2] §3.1). */
      load_row(target, dtype, b * (K + 1) + K, V, lt);
      row_dist(lt, V, T, P, p, scratch, &margin);
      out[K] = (int32_t)inverse_cdf(p, V, (double)u[K], &margin);
    }
    out_accept_len[b] = j;
    if (out_margin) out_margin[b] = margin;
  }
  free(lt); free(ld); free(p); free(q); free(w); free(scratch);
  return 0;
}

int oracle_row_stats(const void* rows, int dtype, int64_t nrows, int64_t V, float temperature, float top_p,
                     double* out) {
  if (!rows || !out || nrows < 0 || V < 1 || (dtype != 0 && dtype != 1)) return -1;
  if (!(temperature > 0.0f) || !(top_p > 0.0f && top_p <= 1.0f)) return -1;
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  val_idx* scratch = (val_idx*)malloc(sizeof(val_idx) * (size_t)V);
  if (!l || !p || !scratch) {
    free(l); free(p); free(scratch);
    return -1;
  }
  for (int64_t r = 0; r < nrows; ++r) {
    load_row(rows, dtype, r, V, l);
    double M, lse, PS = 1.0, tau = -INFINITY;
    softmax_T(l, V, (double)temperature, p, &M, &lse);
    if (top_p < 1.0f) nucleus(l, p, V, (double)top_p, scratch, &PS, &tau, NULL);
    out[4 * r + 0] = M;
    out[4 * r + 1] = lse;
    out[4 * r + 2] = PS;
    out[4 * r + 3] = tau;
  }
  free(l); free(p); free(scratch);
  return 0;
}

/* ------------------------------------------------------------- greedy */

int oracle_verify_greedy(const void* logits, int dtype, const int32_t* cand, int64_t B, int32_t G, int32_t N,
                         int64_t V, int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_best) {
  if (!logits || !cand || !out_tokens || !out_accept_len) return -1;
  if (B < 0 || G < 1 || N < 2 || V < 2 || (dtype != 0 && dtype != 1)) return -1;
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  int64_t* a = (int64_t*)malloc(sizeof(int64_t) * (size_t)G * (size_t)N);
  if (!l || !a) {
    free(l); free(a);
    return -1;
  }
  for (int64_t b = 0; b < B; ++b) {
    int32_t* out = out_tokens + b * N;
    for (int n = 0; n < N; ++n) out[n] = -1;
    int ok = 1;
    for (int64_t k = 0; k < (int64_t)G * (N - 1); ++k) {
      int32_t c = cand[b * G * (N - 1) + k];
      ok &= (c >= 0 && (int64_t)c < V);
    }
    /* a_{g,n} = argmax of row (g, n), lowest index among equal maxima. */
    for (int g = 0; ok && g < G; ++g)
      for (int n = 0; ok && n < N; ++n) {
        load_row(logits, dtype, (b * G + g) * N + n, V, l);
        if (row_has_nan(l, V)) ok = 0;
        a[g * N + n] = argmax_lowest(l, V);
      }
    if (!ok) {
      out_accept_len[b] = -1;
      if (out_best) out_best[b] = -1;
      continue;
    }
    /* [P4] verify branch: candidate token n must equal the argmax at n; the
     * longest matched prefix wins (lowest g on ties), then one bonus token. */
    int best_g = 0, best_L = -1;
    for (int g = 0; g < G; ++g) {
      const int32_t* c = cand + (b * G + g) * (N - 1);
      int L = 0;
      while (L < N - 1 && (int64_t)c[L] == a[g * N + L]) ++L;
      if (L > best_L) {
        best_L = L;
        best_g = g;
      }
    }
    const int32_t* c = cand + (b * G + best_g) * (N - 1);
    for (int n = 0; n < best_L; ++n) out[n] = c[n];
    out[best_L] = (int32_t)a[best_g * N + best_L];
    out_accept_len[b] = best_L;
    if (out_best) out_best[b] = best_g;
  }
  free(l);
  free(a);
  return 0;
}

/* ------------------------------------------------- Lookahead sampling */

int oracle_verify_lookahead_sample(const void* logits, int dtype, const int32_t* cand, const float* uniforms,
                                   int64_t B, int32_t G, int32_t N, int64_t V, float temperature,
                                   int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_best,
                                   double* out_margin) {
  if (!logits || !cand || !uniforms || !out_tokens || !out_accept_len) return -1;
  if (B < 0 || G < 1 || N < 2 || V < 2 || (dtype != 0 && dtype != 1)) return -1;
  if (!(temperature > 0.0f)) return -1;
  const double T = (double)temperature;
  const int64_t NU = (int64_t)(N - 1) * G + 1; /* uniforms per sequence */
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int* alive = (int*)malloc(sizeof(int) * (size_t)G);
  if (!l || !p || !w || !alive) {
    free(l); free(p); free(w); free(alive);
    return -1;
  }
  for (int64_t b = 0; b < B; ++b) {
    int32_t* out = out_tokens + b * N;
    const int32_t* c = cand + b * G * (N - 1); /* c[g*(N-1) + n] */
    const float* u = uniforms + b * NU;
    double margin = INFINITY;
    for (int n = 0; n < N; ++n) out[n] = -1;

    /* Input checks cover every candidate id, every uniform and every row of
     * the sequence, whichever the walk later reaches. */
    int ok = 1;
    for (int64_t k = 0; k < (int64_t)G * (N - 1); ++k) ok &= (c[k] >= 0 && (int64_t)c[k] < V);
    for (int64_t k = 0; k < NU; ++k) ok &= (u[k] >= 0.0f && u[k] < 1.0f);
    for (int64_t r = 0; ok && r < (int64_t)G * N; ++r) {
      load_row(logits, dtype, b * G * N + r, V, l);
      ok = row_ok_sampling(l, V);
    }
    if (!ok) {
      out_accept_len[b] = -1;
      if (out_best) out_best[b] = -1;
      if (out_margin) out_margin[b] = INFINITY;
      continue;
    }

    for (int g = 0; g < G; ++g) alive[g] = 1;
    int lead = 0, j = N - 1;
    for (int n = 0; n < N - 1; ++n) {
      /* The distribution at position n is the owning candidate's row. */
      load_row(logits, dtype, (b * G + lead) * N + n, V, l);
      softmax_T(l, V, T, p, NULL, NULL);
      int accepted = -1;
      for (int g = 0; g < G; ++g) {
        if (!alive[g]) continue;
        const int32_t x = c[g * (N - 1) + n];
        /* q is one-hot on x, so alpha = min(1, p(x)/1) = p(x). */
        const double alpha = p[x];
        if (alpha > 0.0) {
          double du = fabs((double)u[n * G + g] - alpha);
          if (du < margin) margin = du;
        }
        if ((double)u[n * G + g] < alpha) {
          accepted = g;
          break;
        }
        /* Rejected: p <- norm(max(0, p - onehot(x))). A zero residual cannot
         * follow a rejection (it needs p(x) = 1, which always accepts); if
         * rounding ever gave one, p is kept, as the pages fall back to p. */
        double Z = 0.0;
        for (int64_t v = 0; v < V; ++v) {
          w[v] = fmax(0.0, p[v] - (v == x ? 1.0 : 0.0));
          Z += w[v];
        }
        if (Z > 0.0)
          for (int64_t v = 0; v < V; ++v) p[v] = w[v] / Z;
      }
      if (accepted < 0) {
        out[n] = (int32_t)inverse_cdf(p, V, (double)u[(N - 1) * G], &margin);
        j = n;
        break;
      }
      const int32_t x = c[accepted * (N - 1) + n];
      out[n] = x;
      for (int g = 0; g < G; ++g) alive[g] = alive[g] && (c[g * (N - 1) + n] == x);
      lead = accepted;
    }
    if (j == N - 1) {
      /* Every position accepted: the bonus from the owner's last row. */
      load_row(logits, dtype, (b * G + lead) * N + (N - 1), V, l);
      softmax_T(l, V, T, p, NULL, NULL);
      out[N - 1] = (int32_t)inverse_cdf(p, V, (double)u[(N - 1) * G], &margin);
    }
    out_accept_len[b] = j;
    if (out_best) out_best[b] = lead;
    if (out_margin) out_margin[b] = margin;
  }
  free(l); free(p); free(w); free(alive);
  return 0;
}

/* ------------------------------------------------ multi-draft sampling */

int oracle_verify_multidraft_sample(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                                    const float* uniforms, int64_t B, int32_t G, int32_t N, int64_t V,
                                    float temperature, int32_t* out_tokens, int32_t* out_accept_len,
                                    int32_t* out_best, double* out_margin) {
  if (!target || !draft || !draft_tokens || !uniforms || !out_tokens || !out_accept_len) return -1;
  if (B < 0 || G < 1 || N < 2 || V < 2 || (dtype != 0 && dtype != 1)) return -1;
  if (!(temperature > 0.0f)) return -1;
  const double T = (double)temperature;
  const int64_t NU = (int64_t)(N - 1) * G + 1;
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int* alive = (int*)malloc(sizeof(int) * (size_t)G);
  if (!l || !p || !q || !w || !alive) {
    free(l); free(p); free(q); free(w); free(alive);
    return -1;
  }
  for (int64_t b = 0; b < B; ++b) {
    int32_t* out = out_tokens + b * N;
    const int32_t* x = draft_tokens + b * G * (N - 1); /* x[g*(N-1) + n] */
    const float* u = uniforms + b * NU;
    double margin = INFINITY;
    for (int n = 0; n < N; ++n) out[n] = -1;

    int ok = 1;
    for (int64_t k = 0; k < (int64_t)G * (N - 1); ++k) ok &= (x[k] >= 0 && (int64_t)x[k] < V);
    for (int64_t k = 0; k < NU; ++k) ok &= (u[k] >= 0.0f && u[k] < 1.0f);
    for (int64_t r = 0; ok && r < (int64_t)G * N; ++r) {
      load_row(target, dtype, b * G * N + r, V, l);
      ok = row_ok_sampling(l, V);
    }
    for (int64_t r = 0; ok && r < (int64_t)G * (N - 1); ++r) {
      load_row(draft, dtype, b * G * (N - 1) + r, V, l);
      ok = row_ok_sampling(l, V);
    }
    if (!ok) {
      out_accept_len[b] = -1;
      if (out_best) out_best[b] = -1;
      if (out_margin) out_margin[b] = INFINITY;
      continue;
    }

    for (int g = 0; g < G; ++g) alive[g] = 1;
    int lead = 0, j = N - 1;
    for (int n = 0; n < N - 1; ++n) {
      load_row(target, dtype, (b * G + lead) * N + n, V, l);
      softmax_T(l, V, T, p, NULL, NULL);
      int accepted = -1;
      for (int g = 0; g < G; ++g) {
        if (!alive[g]) continue;
        const int32_t xg = x[g * (N - 1) + n];
        load_row(draft, dtype, (b * G + g) * (N - 1) + n, V, l);
        softmax_T(l, V, T, q, NULL, NULL); /* q_g, the distribution x_g came from */
        const double px = p[xg], qx = q[xg];
        double alpha;
        if (px == 0.0)
          alpha = 0.0;
        else if (qx == 0.0)
          alpha = 1.0;
        else
          alpha = fmin(1.0, px / qx);
        if (alpha > 0.0) {
          double du = fabs((double)u[n * G + g] - alpha);
          if (du < margin) margin = du;
        }
        if ((double)u[n * G + g] < alpha) {
          accepted = g;
          break;
        }
        /* Rejected: p <- norm(max(0, p - q_g)), or p itself if that is all zero. */
        double Z = 0.0;
        for (int64_t v = 0; v < V; ++v) {
          w[v] = fmax(0.0, p[v] - q[v]);
          Z += w[v];
        }
        if (Z > 0.0)
          for (int64_t v = 0; v < V; ++v) p[v] = w[v] / Z;
      }
      if (accepted < 0) {
        out[n] = (int32_t)inverse_cdf(p, V, (double)u[(N - 1) * G], &margin);
        j = n;
        break;
      }
      const int32_t xa = x[accepted * (N - 1) + n];
      out[n] = xa;
      for (int g = 0; g < G; ++g) alive[g] = alive[g] && (x[g * (N - 1) + n] == xa);
      lead = accepted;
    }
    if (j == N - 1) {
      load_row(target, dtype, (b * G + lead) * N + (N - 1), V, l);
      softmax_T(l, V, T, p, NULL, NULL);
      out[N - 1] = (int32_t)inverse_cdf(p, V, (double)u[(N - 1) * G], &margin);
    }
    out_accept_len[b] = j;
    if (out_best) out_best[b] = lead;
    if (out_margin) out_margin[b] = margin;
  }
  free(l); free(p); free(q); free(w); free(alive);
  return 0;
}

/* ------------------------------------------------- LM head + verify */

int oracle_verify_sample_lmhead(const void* h_target, const void* h_draft, const void* w_target, const void* w_draft,
                                int dtype, const int32_t* draft_tokens, const float* uniforms, int64_t B, int32_t K,
                                int64_t D, int64_t V, float temperature, float top_p, int32_t* out_tokens,
                                int32_t* out_accept_len, double* out_margin) {
  if (!h_target || !h_draft || !w_target || !w_draft) return -1;
  if (B < 0 || K < 1 || D < 1 || V < 2 || (dtype != 0 && dtype != 1)) return -1;
  double* lt = (double*)malloc(sizeof(double) * (size_t)(B * (K + 1) * V + 1));
  double* ld = (double*)malloc(sizeof(double) * (size_t)(B * K * V + 1));
  if (!lt || !ld) {
    free(lt); free(ld);
    return -1;
  }
  /* logits[r, v] = sum_d h[r, d] * W[v, d], each product and sum in fp64. */
  for (int64_t r = 0; r < B * (K + 1); ++r)
    for (int64_t v = 0; v < V; ++v) {
      double s = 0.0;
      for (int64_t d = 0; d < D; ++d) s += load_logit(h_target, dtype, r * D + d) * load_logit(w_target, dtype, v * D + d);
      lt[r * V + v] = s;
    }
  for (int64_t r = 0; r < B * K; ++r)
    for (int64_t v = 0; v < V; ++v) {
      double s = 0.0;
      for (int64_t d = 0; d < D; ++d) s += load_logit(h_draft, dtype, r * D + d) * load_logit(w_draft, dtype, v * D + d);
      ld[r * V + v] = s;
    }
  const int rc = oracle_verify_sample(lt, ld, 2, draft_tokens, uniforms, B, K, V, temperature, top_p, out_tokens,
                                      out_accept_len, out_margin);
  free(lt);
  free(ld);
  return rc;
}

/* ------------------------------------------------- test-only entry points */

int oracle_inverse_cdf(const double* w, int64_t V, double u, int64_t* out_token) {
  if (!w || !out_token || V < 1) return -1;
  *out_token = inverse_cdf(w, V, u, NULL);
  return 0;
}

int oracle_residual_draw(const double* p, const double* q, int64_t V, double u, int64_t* out_token) {
  if (!p || !q || !out_token || V < 1) return -1;
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  if (!w) return -1;
  *out_token = residual_draw(p, q, w, V, u, NULL);
  free(w);
  return 0;
}

/* ------------------------------------------------------------ n-gram pool */
/* [P4] section "N-gram 池与身份判定": a pool caches the n-grams the lookahead
 * branch collects (W new n-grams of N tokens per step, section "Lookahead
 * 分支:用 2D 窗口制造 n-gram"); only n-grams whose first token equals the
 * last generated token are verified, at most G of them (the "GUESS_SET_SIZE"
 * of the engineering section), and n-grams that are not adopted stay in the
 * pool. The page leaves open how much the pool holds and what it drops; the
 * readings taken: each sequence has its own pool; each first token keeps at
 * most `cap` n-grams; the n-grams of a step are inserted in order; an n-gram
 * already held is not inserted again and keeps its place; inserting into a
 * full key drops that key's oldest n-gram; the candidates are the newest
 * first; an n-gram holding a token outside [0, V) is ignored. The pool here is
 * a plain list per sequence, searched linearly. */

typedef struct {
  int32_t key;
  int32_t* toks; /* the N-1 tokens after the first */
  int64_t stamp; /* insertion order */
} og_entry;

typedef struct {
  og_entry* e;
  int64_t n, cap_alloc;
} og_list;

struct oracle_ngram_pool {
  int64_t B, V;
  int32_t N, cap;
  int64_t next_stamp;
  og_list* seq;
};

oracle_ngram_pool* oracle_ngram_pool_create(int64_t B, int64_t V, int32_t N, int32_t cap) {
  if (B < 0 || V < 1 || N < 2 || cap < 1) return NULL;
  oracle_ngram_pool* p = (oracle_ngram_pool*)calloc(1, sizeof(oracle_ngram_pool));
  if (!p) return NULL;
  p->B = B;
  p->V = V;
  p->N = N;
  p->cap = cap;
  p->seq = (og_list*)calloc((size_t)(B > 0 ? B : 1), sizeof(og_list));
  return p;
}

void oracle_ngram_pool_destroy(oracle_ngram_pool* p) {
  if (!p) return;
  for (int64_t b = 0; b < p->B; ++b) {
    for (int64_t i = 0; i < p->seq[b].n; ++i) free(p->seq[b].e[i].toks);
    free(p->seq[b].e);
  }
  free(p->seq);
  free(p);
}

/* Removes entry i of list l. */
static void og_remove(og_list* l, int64_t i) {
  free(l->e[i].toks);
  for (int64_t k = i + 1; k < l->n; ++k) l->e[k - 1] = l->e[k];
  l->n -= 1;
}

int oracle_ngram_pool_insert(oracle_ngram_pool* p, const int32_t* ngrams, int32_t W) {
  if (!p || (W > 0 && !ngrams) || W < 0) return -1;
  const int32_t N = p->N;
  for (int64_t b = 0; b < p->B; ++b) {
    og_list* l = &p->seq[b];
    for (int32_t w = 0; w < W; ++w) {
      const int32_t* g = ngrams + (b * W + w) * N;
      int ok = 1;
      for (int32_t t = 0; t < N; ++t)
        if (g[t] < 0 || (int64_t)g[t] >= p->V) ok = 0;
      if (!ok) continue; /* a token outside [0, V): ignored */
      /* already held under its first token? */
      int dup = 0;
      int64_t held = 0, oldest = -1;
      for (int64_t i = 0; i < l->n; ++i) {
        if (l->e[i].key != g[0]) continue;
        held += 1;
        if (oldest < 0 || l->e[i].stamp < l->e[oldest].stamp) oldest = i;
        if (memcmp(l->e[i].toks, g + 1, sizeof(int32_t) * (size_t)(N - 1)) == 0) dup = 1;
      }
      if (dup) continue;
      if (held >= p->cap) og_remove(l, oldest); /* a full key drops its oldest n-gram */
      if (l->n == l->cap_alloc) {
        int64_t nc = l->cap_alloc ? 2 * l->cap_alloc : 16;
        og_entry* ne = (og_entry*)realloc(l->e, sizeof(og_entry) * (size_t)nc);
        if (!ne) return -1;
        l->e = ne;
        l->cap_alloc = nc;
      }
      og_entry* e = &l->e[l->n++];
      e->key = g[0];
      e->toks = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N - 1));
      memcpy(e->toks, g + 1, sizeof(int32_t) * (size_t)(N - 1));
      e->stamp = p->next_stamp++;
    }
  }
  return 0;
}

int oracle_ngram_pool_lookup(const oracle_ngram_pool* p, const int32_t* last, int32_t G, int32_t* cand,
                             int32_t* count) {
  if (!p || !last || !cand || !count || G < 1) return -1;
  const int32_t N = p->N;
  for (int64_t b = 0; b < p->B; ++b) {
    int32_t* out = cand + b * (int64_t)G * (N - 1);
    const int32_t key = last[b];
    if (key < 0 || (int64_t)key >= p->V) {
      for (int64_t k = 0; k < (int64_t)G * (N - 1); ++k) out[k] = -1;
      count[b] = -1;
      continue;
    }
    /* the first-token filter, newest first: repeatedly take the unused entry
     * with the largest stamp */
    const og_list* l = &p->seq[b];
    int64_t prev = INT64_MAX;
    int32_t c = 0;
    while (c < G) {
      int64_t best = -1;
      for (int64_t i = 0; i < l->n; ++i)
        if (l->e[i].key == key && l->e[i].stamp < prev && (best < 0 || l->e[i].stamp > l->e[best].stamp)) best = i;
      if (best < 0) break;
      memcpy(out + (int64_t)c * (N - 1), l->e[best].toks, sizeof(int32_t) * (size_t)(N - 1));
      prev = l->e[best].stamp;
      c += 1;
    }
    count[b] = c;
    /* unused slots: a copy of the newest candidate, or, with none, the last
     * token repeated (any guess keeps the greedy verify exact) */
    for (int32_t g = c; g < G; ++g)
      for (int32_t t = 0; t < N - 1; ++t) out[(int64_t)g * (N - 1) + t] = c > 0 ? out[t] : key;
  }
  return 0;
}
