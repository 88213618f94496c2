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
 *        matched prefix wins, plus one bonus token).
 *
 * Dtype codes: 0 = fp32, 1 = bf16 (raw 16-bit patterns).
 * Return value of every function: 0 on success, -1 on an argument error.
 * Per-sequence input errors (token id outside [0,V), uniform outside [0,1),
 * NaN logit, +inf logit or an all -inf row in sampling mode, NaN in greedy
 * mode) give out_accept_len[b] = -1 and out_tokens[b,:] = -1.
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

#ifdef __cplusplus
}
#endif
#endif
