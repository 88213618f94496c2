/*
 * oracle.h — plain CPU reference of the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY. This code exists to check the GPU library. Only
 * the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg may load or call it. The GPU library never links, includes or calls it,
 * and shares no code with it.
 *
 * Everything is computed in fp64, single-threaded, one sequence at a time,
 * in the order the pages give the algorithm. Sources (page title, section):
 *   [P1] "Speculative Decoding —— LLM推理优化技术（一）", §2.1 (accept
 *        probability and residual distribution), §2.2 (proof that the output
 *        follows p), §2.3 (sequential test, stop at the first rejection,
 *        bonus token), §4 (temperature on both sides; the residual falls back
 *        to p when it sums to zero; p/(q+eps) ratio).
 *   [P2] kwkr.cn "投机解码", §3.1 (r < alpha accepts, r >= alpha rejects;
 *        renormalise the residual; bonus token), §3.2 (fp32 or better for
 *        the probabilities), §3.4 (temperature and top-p identical on both
 *        sides; resample only inside the truncated set).
 *   [P4] "Lookahead Decoding 完全拆解", section "验证分支" (greedy verify:
 *        candidate token i must equal the argmax at position i; longest
 *        matched prefix wins, plus one bonus token) and section
 *        "采样模式的验证" (sampling-mode verify of greedily produced
 *        candidates: the draft distribution is one-hot on the token).
 *
 * Dtype codes: 0 = fp32, 1 = bf16 (raw 16-bit patterns); the sampling verify
 * also takes 2 = fp64, for logits the oracle computes itself.
 * Return value of every function: 0 on success, -1 on an argument error.
 * Per-sequence input errors (token id outside [0,V), uniform outside [0,1),
 * NaN logit, +inf logit or an all -inf row in the sampling modes, NaN in
 * greedy mode) give out_accept_len[b] = -1 and out_tokens[b,:] = -1.
 */
#ifndef SPECVERIFY_ORACLE_H
#define SPECVERIFY_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Sampling-mode verify.
 *   target [B,K+1,V], draft [B,K,V] (row i of target tests draft token i;
 *   target row K is the bonus distribution); draft_tokens [B,K];
 *   uniforms [B,K+1] (u_0..u_{K-1} accept tests, u_K drives the one sample).
 *   temperature >= 0 (0 = greedy limit: argmax match, uniforms unused);
 *   top_p in (0,1] (1 = no filter).
 * Outputs: out_tokens [B,K+1] (accepted prefix, then the resampled or bonus
 *   token, then -1), out_accept_len [B] in [0,K].
 *   out_margin [B] (nullable): the smallest distance to a decision boundary
 *   met in that sequence: |u_i - alpha_i| for each accept test, the gap of
 *   u_K*Z to the edges of the sampled token's CDF interval divided by Z, and
 *   for each nucleus used, the distance of top_p to the cumulative masses on
 *   either side of the cut. +inf when no such decision was taken. */
int oracle_verify_sample(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                         const float* uniforms, int64_t B, int32_t K, int64_t V, float temperature, float top_p,
                         int32_t* out_tokens, int32_t* out_accept_len, double* out_margin);

/* Per-row normalisers, for rows [nrows, V]: out [nrows, 4] =
 *   { m = max_v l_v/T, lse = log sum_v exp(l_v/T), P_S = nucleus mass
 *     (1 when top_p == 1), tau = stored logit value at the nucleus cut
 *     (-inf when top_p == 1) }.  temperature must be > 0. */
int oracle_row_stats(const void* rows, int dtype, int64_t nrows, int64_t V, float temperature, float top_p,
                     double* out);

/* Greedy (Lookahead) verify. logits [B,G,N,V], cand [B,G,N-1].
 * out_tokens [B,N]: matched prefix of the best candidate, then its bonus
 * token (the argmax after the prefix), then -1. out_accept_len [B] in
 * [0,N-1]. out_best [B] (nullable): the winning candidate, lowest g on ties. */
int oracle_verify_greedy(const void* logits, int dtype, const int32_t* cand, int64_t B, int32_t G, int32_t N,
                         int64_t V, int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_best);

/* Lookahead sampling-mode verify ([P4] section "采样模式的验证"): the
 * candidates were produced greedily, so each one's draft distribution is
 * one-hot on its token and only the token id is kept. logits [B,G,N,V]: row
 * (g, n) is the target distribution at position n of candidate g's branch;
 * cand [B,G,N-1]; uniforms [B,(N-1)*G+1]: u[n*G+g] is the accept test of
 * candidate g at position n, u[(N-1)*G] drives the one draw; temperature > 0.
 * At each position the still-matching candidates are tested in order of g
 * against the current distribution, which starts as softmax(row/T) of the
 * candidate that owns the accepted prefix (g = 0 at position 0). Candidate x
 * is accepted when u < p(x) (alpha = min(1, p(x)/q(x)) with q one-hot); a
 * rejection replaces p by norm(max(0, p - onehot(x))), i.e. p with x removed.
 * When no candidate is accepted at position n, the token is drawn from the
 * current p and the round ends; when all N-1 positions are accepted the bonus
 * is drawn from row N-1 of the owning candidate.
 * out_tokens [B,N] (accepted prefix, drawn token, -1 tail); out_accept_len
 * [B] in [0,N-1]; out_best [B] (nullable): the candidate that owns the
 * accepted prefix; out_margin [B] (nullable): as in oracle_verify_sample. */
int oracle_verify_lookahead_sample(const void* logits, int dtype, const int32_t* cand, const float* uniforms,
                                   int64_t B, int32_t G, int32_t N, int64_t V, float temperature,
                                   int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_best,
                                   double* out_margin);

/* Multi-draft sampling verify: the same walk with G drafts that were sampled
 * from full draft distributions. draft [B,G,N-1,V]: row (g, n) is the draft
 * distribution (as logits) that draft g's token at position n was drawn from;
 * draft_tokens [B,G,N-1]. Draft g is tested against the current p with
 * alpha = min(1, p(x)/q_g(x)) (q_g(x) = 0 < p(x) gives 1, p(x) = 0 gives 0);
 * a rejection replaces p by norm(max(0, p - q_g)) ([P1] §2.1 applied once per
 * rejected draft; if that is all zero, p is kept, [P1] §4). Temperature
 * applies to both sides ([P2] §3.4). Everything else — the owner's rows, the
 * prefix filter, the uniform layout, the draw, the outputs and the input
 * checks (every draft row too) — is as in oracle_verify_lookahead_sample. */
int oracle_verify_multidraft_sample(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                                    const float* uniforms, int64_t B, int32_t G, int32_t N, int64_t V,
                                    float temperature, int32_t* out_tokens, int32_t* out_accept_len,
                                    int32_t* out_best, double* out_margin);

/* The sampling verify on logits computed from hidden states by the LM heads:
 * target logits [B,K+1,V] = h_target [B,K+1,D] · w_target[V,D]^T, draft
 * logits [B,K,V] = h_draft [B,K,D] · w_draft[V,D]^T, every product and sum in
 * fp64 (no rounding to a stored logit type), then oracle_verify_sample on
 * them. This is the computation a fused LM-head GEMM with a verify epilogue
 * must reproduce; the pages' verify takes the logits as given. dtype 0 or 1
 * for h and w. */
int oracle_verify_sample_lmhead(const void* h_target, const void* h_draft, const void* w_target, const void* w_draft,
                                int dtype, const int32_t* draft_tokens, const float* uniforms, int64_t B, int32_t K,
                                int64_t D, int64_t V, float temperature, float top_p, int32_t* out_tokens,
                                int32_t* out_accept_len, double* out_margin);

/* N-gram pool ([P4] section "N-gram 池与身份判定"): one pool per sequence,
 * keyed by an n-gram's first token, each key holding at most `cap` n-grams
 * of N tokens.
 *   create/destroy: an empty pool for B sequences over a vocabulary of V.
 *   insert: ngrams [B, W, N]; sequence b's W n-grams go into its pool in
 *     order. An n-gram already held is not inserted again; a full key drops
 *     its oldest n-gram; an n-gram with a token outside [0, V) is ignored.
 *   lookup: for each b, the n-grams whose first token equals last[b], newest
 *     first, at most G: cand [B, G, N-1] holds their tokens after the first,
 *     count [B] how many there are. Unused slots hold a copy of the newest
 *     candidate, or last[b] repeated when there is none. A last token outside
 *     [0, V) gives count -1 and -1 tokens. The pool is not changed. */
typedef struct oracle_ngram_pool oracle_ngram_pool;
oracle_ngram_pool* oracle_ngram_pool_create(int64_t B, int64_t V, int32_t N, int32_t cap);
void oracle_ngram_pool_destroy(oracle_ngram_pool* p);
int oracle_ngram_pool_insert(oracle_ngram_pool* p, const int32_t* ngrams, int32_t W);
int oracle_ngram_pool_lookup(const oracle_ngram_pool* p, const int32_t* last, int32_t G, int32_t* cand,
                             int32_t* count);

/* Test-only entry points to the draw's two edge rules, so that tests can pin
 * them directly (valid verify inputs do not reach them in exact arithmetic).
 * oracle_inverse_cdf: the inverse-CDF draw from unnormalised weights w[V]:
 *   the smallest t with sum_{v<=t} w_v > u * sum_v w_v; if u * Z is at or past
 *   the last partial sum, the largest t with w_t > 0.
 * oracle_residual_draw: the draw after a rejection, from max(0, p - q), or
 *   from p when that residual is all zero ([P1] §4). */
int oracle_inverse_cdf(const double* w, int64_t V, double u, int64_t* out_token);
int oracle_residual_draw(const double* p, const double* q, int64_t V, double u, int64_t* out_token);

#ifdef __cplusplus
}
#endif
#endif
