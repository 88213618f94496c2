/*
 * specgen — seeded synthetic inputs for the speculative-decoding verify step.
 *
 * This module produces inputs only. It is shared by the CPU oracle's tests and
 * by the GPU benchmark so that both see identical bytes; it contains none of
 * the verify step's arithmetic (no accept test, no residual, no normaliser
 * that the verifier would reuse).
 *
 * Random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11), written here from the published
 * round function. Each quantity draws from its own stream (a key), and the
 * counter is the flat index of the element it belongs to, so the bytes do not
 * depend on the thread count or on how the batch is split across processes.
 *
 * Workload shapes follow the synthetic configurations of the verify step:
 *   target logits  l_t = sigma_t * N(0,1) (+ peak height at n_peaks distinct
 *                  random indices per row), rounded to the storage type last;
 *   draft logits   l_d = l_t (before rounding) + sigma_d * N(0,1), rounded;
 *   draft tokens   one draw from the draft model's sampling distribution
 *                  softmax(l_d / T), restricted to the top-p nucleus when
 *                  top_p < 1. This stands in for the draft model's own sampler
 *                  (which the pages write as torch.multinomial over
 *                  softmax(logits / T)); it uses the Gumbel-max trick, which
 *                  the verifier never uses;
 *   uniforms       U(0,1) fp32, one per accept test plus one for the sample;
 *   greedy         logits sigma * N(0,1); candidate token t equals its row's
 *                  argmax with probability match_prob per step until the first
 *                  miss, then uniform random ids (the Lookahead n-gram stand-in).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- Philox */

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static inline void mulhilo32(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  *hi = (uint32_t)(p >> 32);
  *lo = (uint32_t)p;
}

/* One Philox4x32 round followed by the key schedule, ten times. */
void sg_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint32_t hi0, lo0, hi1, lo1;
    mulhilo32(PHILOX_M0, c0, &hi0, &lo0);
    mulhilo32(PHILOX_M1, c2, &hi1, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Stream identifiers: one key per quantity. */
enum {
  SG_S_TARGET = 1,  /* target logit noise, counter = flat target element   */
  SG_S_DRAFT = 2,   /* draft logit noise, counter = flat draft element     */
  SG_S_PEAK = 3,    /* peak positions, counter = (global row, attempt)     */
  SG_S_GUMBEL = 4,  /* draft sampler noise, counter = flat draft element   */
  SG_S_UNIFORM = 5, /* verify uniforms, counter = flat uniform index       */
  SG_S_GREEDY = 6,  /* greedy logits, counter = flat element               */
  SG_S_CAND = 7     /* greedy candidates, counter = flat candidate slot    */
};

static inline void sg_key(uint64_t seed, uint32_t stream, uint32_t key[2]) {
  key[0] = (uint32_t)seed;
  key[1] = (uint32_t)(seed >> 32) ^ (0x5EED0000u | stream);
}

static inline void sg_draw(uint64_t seed, uint32_t stream, uint64_t idx, uint32_t sub, uint32_t out[4]) {
  uint32_t key[2];
  sg_key(seed, stream, key);
  uint32_t ctr[4] = {(uint32_t)idx, (uint32_t)(idx >> 32), sub, 0u};
  sg_philox4x32_10(ctr, key, out);
}

/* Standard normal by Box-Muller from two 32-bit words (u1 in (0,1], u2 in [0,1)). */
static inline double sg_normal(uint64_t seed, uint32_t stream, uint64_t idx) {
  uint32_t r[4];
  sg_draw(seed, stream, idx, 0u, r);
  double u1 = ((double)r[0] + 1.0) * (1.0 / 4294967296.0);
  double u2 = (double)r[1] * (1.0 / 4294967296.0);
  return sqrt(-2.0 * log(u1)) * cos(2.0 * M_PI * u2);
}

/* U(0,1) as fp32 with 24 random bits: exactly representable, in [0,1). */
static inline float sg_uniform24(uint32_t r) { return (float)(r >> 8) * (1.0f / 16777216.0f); }

/* Uniform integer in [0, n) by 32x64 multiply-shift. */
static inline uint64_t sg_below(uint32_t r, uint64_t n) { return ((uint64_t)r * n) >> 32; }

/* fp32 -> bf16 bits, round to nearest even; NaN stays a quiet NaN. */
static inline uint16_t sg_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static inline float sg_from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static inline float sg_load(const void* base, int dtype, uint64_t i) {
  return dtype == 1 ? sg_from_bf16(((const uint16_t*)base)[i]) : ((const float*)base)[i];
}

static inline void sg_store(void* base, int dtype, uint64_t i, float v) {
  if (dtype == 1)
    ((uint16_t*)base)[i] = sg_to_bf16(v);
  else
    ((float*)base)[i] = v;
}

/* ----------------------------------------------------------- thread pool */

typedef void (*sg_range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct {
  sg_range_fn fn;
  void* ctx;
  int64_t lo, hi;
} sg_job;

static void* sg_job_main(void* p) {
  sg_job* j = (sg_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void sg_parallel(int64_t n, int nthreads, sg_range_fn fn, void* ctx) {
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  pthread_t th[256];
  sg_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].lo = n * t / nthreads;
    jobs[t].hi = n * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, sg_job_main, &jobs[t]) != 0) break;
    started = t;
  }
  sg_job_main(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  for (int t = started + 1; t < nthreads; ++t) sg_job_main(&jobs[t]); /* threads that failed to start */
}

/* ------------------------------------------------------------- logits */

typedef struct {
  void* target;
  void* draft; /* may be NULL */
  int dtype;
  int64_t B, K, V;
  double target_sigma, peak_height, draft_sigma;
  int n_peaks;
  uint64_t seed;
  int64_t seq_offset;
} sg_logits_ctx;

static void sg_logits_range(void* p, int64_t lo, int64_t hi) {
  sg_logits_ctx* c = (sg_logits_ctx*)p;
  const int64_t V = c->V, K = c->K;
  float* row = (float*)malloc(sizeof(float) * (size_t)V);
  int64_t* peaks = (int64_t*)malloc(sizeof(int64_t) * (size_t)(c->n_peaks > 0 ? c->n_peaks : 1));
  for (int64_t b = lo; b < hi; ++b) {
    const int64_t bg = c->seq_offset + b;
    for (int64_t i = 0; i <= K; ++i) {
      const uint64_t rg = (uint64_t)(bg * (K + 1) + i); /* global target row */
      for (int64_t v = 0; v < V; ++v) row[v] = (float)(c->target_sigma * sg_normal(c->seed, SG_S_TARGET, rg * (uint64_t)V + (uint64_t)v));
      int np = c->n_peaks < V ? c->n_peaks : (int)V;
      int have = 0;
      for (uint32_t attempt = 0; have < np && attempt < 1000000u; ++attempt) {
        uint32_t r[4];
        sg_draw(c->seed, SG_S_PEAK, rg, attempt, r);
        int64_t idx = (int64_t)sg_below(r[0], (uint64_t)V);
        int dup = 0;
        for (int q = 0; q < have; ++q) dup |= (peaks[q] == idx);
        if (!dup) peaks[have++] = idx;
      }
      for (int q = 0; q < have; ++q) row[peaks[q]] = (float)((double)row[peaks[q]] + c->peak_height);
      const uint64_t tb = (uint64_t)((b * (K + 1) + i) * V);
      for (int64_t v = 0; v < V; ++v) sg_store(c->target, c->dtype, tb + (uint64_t)v, row[v]);
      if (c->draft && i < K) {
        const uint64_t dg = (uint64_t)(bg * K + i); /* global draft row */
        const uint64_t db = (uint64_t)((b * K + i) * V);
        for (int64_t v = 0; v < V; ++v) {
          double n = sg_normal(c->seed, SG_S_DRAFT, dg * (uint64_t)V + (uint64_t)v);
          sg_store(c->draft, c->dtype, db + (uint64_t)v, (float)((double)row[v] + c->draft_sigma * n));
        }
      }
    }
  }
  free(peaks);
  free(row);
}

/* Target [B,K+1,V] and draft [B,K,V] logits. draft may be NULL. */
int sg_gen_logits(void* target, void* draft, int dtype, int64_t B, int32_t K, int64_t V, double target_sigma,
                  double peak_height, int32_t n_peaks, double draft_sigma, uint64_t seed, int64_t seq_offset,
                  int32_t nthreads) {
  if (!target || B < 0 || K < 0 || V < 1 || (dtype != 0 && dtype != 1) || n_peaks < 0) return -1;
  sg_logits_ctx c = {target, draft, dtype, B, K, V, target_sigma, peak_height, draft_sigma, n_peaks, seed, seq_offset};
  sg_parallel(B, nthreads, sg_logits_range, &c);
  return 0;
}

/* ------------------------------------------------------- draft sampler */

/* qsort has no context argument; the nucleus sort keys on (value desc, index asc). */
typedef struct {
  float v;
  int64_t i;
} sg_vi;

static int sg_vi_desc(const void* a, const void* b) {
  const sg_vi* x = (const sg_vi*)a;
  const sg_vi* y = (const sg_vi*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

typedef struct {
  const void* draft;
  int dtype;
  int64_t B, K, V;
  float temperature, top_p;
  uint64_t seed;
  int64_t seq_offset;
  int32_t* tokens;
} sg_tok_ctx;

/* The draft model's sampler stand-in: one draw from softmax(l/T) over the
 * nucleus, via Gumbel-max (argmax of l/T + G, G standard Gumbel). The nucleus
 * is the smallest value-threshold set {l >= tau} whose mass reaches top_p,
 * found by sorting; ties at the cut are all kept. T == 0 takes the argmax
 * (lowest index among equal maxima). */
static void sg_tokens_range(void* p, int64_t lo, int64_t hi) {
  sg_tok_ctx* c = (sg_tok_ctx*)p;
  const int64_t V = c->V, K = c->K;
  const int use_nucleus = c->temperature > 0.0f && c->top_p < 1.0f;
  float* row = (float*)malloc(sizeof(float) * (size_t)V);
  sg_vi* order = use_nucleus ? (sg_vi*)malloc(sizeof(sg_vi) * (size_t)V) : NULL;
  for (int64_t b = lo; b < hi; ++b) {
    for (int64_t i = 0; i < K; ++i) {
      const uint64_t base = (uint64_t)((b * K + i) * V);
      for (int64_t v = 0; v < V; ++v) row[v] = sg_load(c->draft, c->dtype, base + (uint64_t)v);
      int64_t best = 0;
      if (c->temperature <= 0.0f) {
        for (int64_t v = 1; v < V; ++v)
          if (row[v] > row[best]) best = v;
      } else {
        const double T = (double)c->temperature;
        double cut = -INFINITY; /* keep v iff row[v] >= cut */
        if (use_nucleus) {
          double mx = -INFINITY;
          for (int64_t v = 0; v < V; ++v) mx = row[v] > mx ? row[v] : mx;
          double tot = 0.0;
          for (int64_t v = 0; v < V; ++v) tot += exp(((double)row[v] - mx) / T);
          for (int64_t v = 0; v < V; ++v) { order[v].v = row[v]; order[v].i = v; }
          qsort(order, (size_t)V, sizeof(sg_vi), sg_vi_desc);
          double acc = 0.0;
          for (int64_t r = 0; r < V; ++r) {
            acc += exp(((double)order[r].v - mx) / T) / tot;
            cut = order[r].v;
            if (acc >= (double)c->top_p) break;
          }
        }
        const uint64_t gflat = (uint64_t)(((c->seq_offset + b) * K + i) * V);
        double bestkey = -INFINITY;
        best = -1;
        for (int64_t v = 0; v < V; ++v) {
          if (!((double)row[v] >= cut) || row[v] == -INFINITY) continue;
          uint32_t r[4];
          sg_draw(c->seed, SG_S_GUMBEL, gflat + (uint64_t)v, 0u, r);
          double u = ((double)r[0] + 0.5) * (1.0 / 4294967296.0); /* (0,1) */
          double key = (double)row[v] / T - log(-log(u));
          if (key > bestkey) { bestkey = key; best = v; }
        }
        if (best < 0) best = 0;
      }
      c->tokens[b * K + i] = (int32_t)best;
    }
  }
  free(order);
  free(row);
}

/* draft_tokens[B,K]: one draw per draft row from the (filtered) draft distribution. */
int sg_draft_tokens(const void* draft, int dtype, int64_t B, int32_t K, int64_t V, float temperature, float top_p,
                    uint64_t seed, int64_t seq_offset, int32_t* tokens, int32_t nthreads) {
  if (!draft || !tokens || B < 0 || K < 0 || V < 1 || (dtype != 0 && dtype != 1)) return -1;
  sg_tok_ctx c = {draft, dtype, B, K, V, temperature, top_p, seed, seq_offset, tokens};
  sg_parallel(B, nthreads, sg_tokens_range, &c);
  return 0;
}

/* uniforms[B,K+1] fp32 in [0,1). */
int sg_uniforms(int64_t B, int32_t K, uint64_t seed, int64_t seq_offset, float* out) {
  if (!out || B < 0 || K < 0) return -1;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t i = 0; i <= K; ++i) {
      uint32_t r[4];
      sg_draw(seed, SG_S_UNIFORM, (uint64_t)((seq_offset + b) * (K + 1) + i), 0u, r);
      out[b * (K + 1) + i] = sg_uniform24(r[0]);
    }
  return 0;
}

/* ------------------------------------------------------------- greedy */

typedef struct {
  void* logits;
  int32_t* cand;
  int dtype;
  int64_t B, G, N, V;
  double sigma, match_prob;
  uint64_t seed;
  int64_t seq_offset;
} sg_greedy_ctx;

static void sg_greedy_range(void* p, int64_t lo, int64_t hi) {
  sg_greedy_ctx* c = (sg_greedy_ctx*)p;
  const int64_t G = c->G, N = c->N, V = c->V;
  for (int64_t b = lo; b < hi; ++b) {
    const int64_t bg = c->seq_offset + b;
    for (int64_t g = 0; g < G; ++g) {
      int missed = 0;
      for (int64_t n = 0; n < N; ++n) {
        const uint64_t rg = (uint64_t)((bg * G + g) * N + n);
        const uint64_t rl = (uint64_t)((b * G + g) * N + n);
        for (int64_t v = 0; v < V; ++v)
          sg_store(c->logits, c->dtype, rl * (uint64_t)V + (uint64_t)v,
                   (float)(c->sigma * sg_normal(c->seed, SG_S_GREEDY, rg * (uint64_t)V + (uint64_t)v)));
        if (n == N - 1) break; /* the last row has no candidate token */
        uint32_t r[4];
        sg_draw(c->seed, SG_S_CAND, (uint64_t)((bg * G + g) * (N - 1) + n), 0u, r);
        int32_t tok;
        if (!missed && (double)r[0] * (1.0 / 4294967296.0) < c->match_prob) {
          int64_t a = 0; /* the stored row's argmax, lowest index among equals */
          float av = sg_load(c->logits, c->dtype, rl * (uint64_t)V);
          for (int64_t v = 1; v < V; ++v) {
            float x = sg_load(c->logits, c->dtype, rl * (uint64_t)V + (uint64_t)v);
            if (x > av) { av = x; a = v; }
          }
          tok = (int32_t)a;
        } else {
          missed = 1;
          tok = (int32_t)sg_below(r[1], (uint64_t)V);
        }
        c->cand[(b * G + g) * (N - 1) + n] = tok;
      }
    }
  }
}

/* logits[B,G,N,V] and cand[B,G,N-1]. */
int sg_gen_greedy(void* logits, int32_t* cand, int dtype, int64_t B, int32_t G, int32_t N, int64_t V, double sigma,
                  double match_prob, uint64_t seed, int64_t seq_offset, int32_t nthreads) {
  if (!logits || !cand || B < 0 || G < 1 || N < 2 || V < 1 || (dtype != 0 && dtype != 1)) return -1;
  sg_greedy_ctx c = {logits, cand, dtype, B, G, N, V, sigma, match_prob, seed, seq_offset};
  sg_parallel(B, nthreads, sg_greedy_range, &c);
  return 0;
}

/* Raw uniforms for tests that need plain U(0,1) doubles from a named stream. */
int sg_uniform_doubles(uint64_t seed, uint32_t stream, uint64_t first, int64_t n, double* out) {
  if (!out || n < 0) return -1;
  for (int64_t k = 0; k < n; ++k) {
    uint32_t r[4];
    sg_draw(seed, stream, first + (uint64_t)k, 0u, r);
    out[k] = ((double)r[0] + 0.5) * (1.0 / 4294967296.0);
  }
  return 0;
}
