/*
 * specverify.h — C ABI of libspecverify, the GB300 (sm_103a) speculative-
 * decoding verify step.
 *
 * The operation. A draft model proposed K tokens x_0..x_{K-1}; the target
 * model scored K+1 positions. Verification turns both models' logits into
 * distributions p (target) and q (draft), accepts x_i while
 * u_i < min(1, p_i(x_i) / q_i(x_i)), stops at the first rejection j, and
 * replaces x_j by a draw from norm(max(0, p_j - q_j)); if all K are accepted
 * it draws one bonus token from p_K. The emitted tokens then follow the target
 * model's distribution exactly. Sources (page title, section):
 *   "Speculative Decoding —— LLM推理优化技术（一）" (hustzhy.cn), §2.1 accept
 *     probability and residual distribution, §2.2 proof, §2.3 sequential test
 *     with a bonus token, §4 temperature on both sides and the fallback to p
 *     when the residual is all zero;
 *   kwkr.cn "投机解码" §3.1 the verify steps (r < alpha accepts), §3.2 fp32
 *     probabilities, §3.4 temperature and top-p applied identically to both
 *     sides, resampling only inside the truncated set;
 *   "Lookahead Decoding 完全拆解" (pinghaoyang.com.cn), verify branch: greedy
 *     verification of n-gram candidates against the per-position argmax,
 *     longest matched prefix plus one bonus token.
 *
 * Conventions shared by every entry point:
 *   - Every array argument is a DEVICE pointer owned by the caller; the
 *     library never frees or retains it past the call's completion on the
 *     stream. Arrays are dense, row-major, with the vocabulary innermost.
 *   - Calls are asynchronous: they validate arguments on the host, enqueue
 *     their kernels on `stream` (one; two for sv_verify_lookahead_sample) (a
 *     cudaStream_t; NULL = the legacy default stream) and return. Results are
 *     valid once the stream reaches them.
 *   - The library keeps a small scratch area per (device, stream), allocated
 *     on the first call that needs it (or a larger one) and reused after.
 *     Calls on the same stream are ordered; calls on different streams use
 *     different scratch areas. sv_release() frees them all.
 *   - Host-checkable errors return a negative sv_status and enqueue nothing.
 *   - Input errors found on the device (a token id outside [0,V), a uniform
 *     outside [0,1), a NaN logit, a +inf logit or an all -inf row in sampling
 *     mode, a NaN logit in greedy mode) mark that sequence only:
 *     out_accept_len[b] = -1 and out_tokens[b,:] = -1. They also set a sticky
 *     flag that sv_get_status() reports. Kernels never trap.
 *   - Every internal wait is bounded; a wait that runs out sets
 *     SV_ERR_TIMEOUT, reported by sv_get_status().
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

typedef enum {
  SV_OK = 0,
  SV_ERR_ARG = -1,     /* bad shape, null pointer, temperature < 0, top_p outside (0,1] */
  SV_ERR_DTYPE = -2,   /* dtype not SV_F32 / SV_BF16, or a misaligned pointer for it */
  SV_ERR_CUDA = -3,    /* a CUDA runtime call failed (launch, allocation, copy) */
  SV_ERR_INPUT = -4,   /* device-detected bad input in at least one sequence */
  SV_ERR_TIMEOUT = -5, /* a bounded device wait ran out; the scratch was reset */
  SV_ERR_NOMEM = -6,   /* scratch allocation failed */
  SV_ERR_SCRATCH_LIMIT = -7 /* sv_verify_sample_noalloc: the call needs more than its fixed scratch */
} sv_status;

/*
 * Sampling-mode verify ("Speculative Decoding" §2.1-2.3; kwkr.cn §3.1, §3.4).
 *
 *   target_logits [B, K+1, V] dtype: row i is the target distribution that
 *                 draft token i is tested against; row K is the bonus
 *                 distribution.
 *   draft_logits  [B, K, V] dtype: row i is the draft distribution that
 *                 produced draft token i. Not read when temperature == 0.
 *   draft_tokens  [B, K] int32.
 *   uniforms      [B, K+1] fp32 in [0,1): u_0..u_{K-1} are the accept tests;
 *                 u_K drives the single inverse-CDF draw (residual or bonus).
 *                 Not read when temperature == 0.
 *   B >= 0, K >= 1, V >= 2; dtype SV_F32 or SV_BF16 (pointers aligned to
 *   the element size).
 *   temperature   > 0: p = softmax(l/T), q likewise, on both sides;
 *                 == 0: the greedy limit: x_i is accepted iff it is the
 *                 argmax of target row i (lowest index among equal maxima);
 *                 at a rejection the token is that argmax; the bonus is the
 *                 argmax of row K.
 *   top_p         in (0,1]; < 1 restricts p and q each to its nucleus — the
 *                 tokens whose stored logit is >= tau, tau the largest value
 *                 whose upper set holds >= top_p of the mass (ties at the cut
 *                 are kept) — and renormalises; 1 = no filter.
 * Outputs:
 *   out_tokens     [B, K+1] int32: x_0..x_{j-1}, then the drawn token at j,
 *                  then -1.
 *   out_accept_len [B] int32: j in [0, K] (-1 for a sequence with bad input).
 *   out_row_stats  nullable [B, 2K+1, 4] fp32, rows in the order target
 *                  0..K, draft 0..K-1: {m = max l/T, lse = log sum exp(l/T),
 *                  P_S = nucleus mass (1 without top-p), tau = stored logit
 *                  at the nucleus cut (-inf without top-p)}. Written only
 *                  when temperature > 0.
 * The selected token is the smallest t with sum_{v<=t} w_v > u_K * sum_v w_v
 * (ascending vocabulary order), w = max(0, p'_j - q'_j) after a rejection
 * (p'_j itself if that is all zero) or p'_K for the bonus.
 */
int sv_verify_sample(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                     const float* uniforms, int64_t B, int32_t K, int64_t V, int32_t dtype, float temperature,
                     float top_p, int32_t* out_tokens, int32_t* out_accept_len, float* out_row_stats,
                     void* stream);

/*
 * Greedy verify of Lookahead n-gram candidates ("Lookahead Decoding 完全拆解",
 * verify branch; "Speculative Decoding" §5.3).
 *
 *   logits [B, G, N, V] dtype: candidate g's N positions (its N-1 tokens and
 *          the bonus position after them).
 *   cand   [B, G, N-1] int32: the candidate n-grams.
 *   B >= 0, G >= 1, N >= 2, V >= 2.
 * a_{g,n} = argmax_v logits[b,g,n,v] (lowest index among equal maxima; -0
 * and +0 are equal). L_g = the longest n with cand[b,g,0..n-1] equal to
 * a_{g,0..n-1}. The winner g* has the largest L_g (lowest g on ties).
 * Outputs:
 *   out_tokens     [B, N] int32: cand[b,g*,0..L-1], then a_{g*,L}, then -1.
 *   out_accept_len [B] int32: L in [0, N-1] (-1 for bad input).
 *   out_best_cand  nullable [B] int32: g*.
 */
int sv_verify_greedy(const void* logits, const int32_t* cand, int64_t B, int32_t G, int32_t N, int64_t V,
                     int32_t dtype, int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_best_cand,
                     void* stream);

/*
 * Sampling-mode verify of Lookahead n-gram candidates ("Lookahead Decoding
 * 完全拆解", section "采样模式的验证"). The candidates were produced greedily,
 * so only their token ids exist: each one's draft distribution is one-hot.
 *
 *   logits   [B, G, N, V] dtype: row (g, n) is the target's distribution
 *            (as logits) at position n of candidate g's branch, i.e. after
 *            cand[b,g,0..n-1]; row N-1 is the bonus position.
 *   cand     [B, G, N-1] int32: the candidate n-grams.
 *   uniforms [B, (N-1)*G + 1] fp32 in [0,1): u[n*G + g] is the accept test of
 *            candidate g at position n (read only if that test happens); the
 *            last one drives the one draw.
 *   B >= 0, 1 <= G <= 32, N >= 2, G*N <= 1024, G*G*(N-1) <= 4096, V >= 2;
 *   B*G*N < 2^31; temperature > 0 (finite).
 * Each position n starts from p = softmax(logits[b, owner, n] / T), where the
 * owner is the candidate whose token was accepted at n-1 (candidate 0 at
 * n = 0). The candidates whose first n tokens equal the accepted prefix are
 * tested in order of g: candidate g's token x is accepted when
 * u[n*G + g] < p(x) (min(1, p(x)/q(x)) with q one-hot; a repeated token has
 * p(x) = 0 by then); a rejection replaces p by p with x removed,
 * renormalised. When none is accepted, the token at n is drawn from the
 * current p and the round ends; after N-1 accepted positions the bonus is
 * drawn from the owner's row N-1. A draw is the smallest t with
 * sum_{v<=t} w_v > u * sum_v w_v (ascending vocabulary order).
 * Outputs:
 *   out_tokens     [B, N] int32: the accepted prefix, the drawn token, -1.
 *   out_accept_len [B] int32: in [0, N-1] (-1 for bad input: a token id
 *                  outside [0,V), a uniform outside [0,1), or a NaN, +inf or
 *                  all -inf row anywhere in the sequence).
 *   out_best_cand  nullable [B] int32: the owner of the accepted prefix.
 *   out_row_lse    nullable [B, G, N] fp32: log sum_v exp(l_v/T) of every row.
 * Two kernels are enqueued on the stream.
 */
int sv_verify_lookahead_sample(const void* logits, const int32_t* cand, const float* uniforms, int64_t B, int32_t G,
                               int32_t N, int64_t V, int32_t dtype, float temperature, int32_t* out_tokens,
                               int32_t* out_accept_len, int32_t* out_best_cand, float* out_row_lse, void* stream);

/*
 * Multi-draft sampling verify: G drafts drawn from full draft distributions,
 * verified by the walk of sv_verify_lookahead_sample with the single-draft
 * rule of "Speculative Decoding —— LLM推理优化技术（一）" §2.1 for each draft.
 *
 *   target       [B, G, N, V] dtype: row (g, n) is the target's distribution
 *                at position n of draft g's branch; row N-1 the bonus.
 *   draft        [B, G, N-1, V] dtype: row (g, n) is the distribution draft
 *                g's token at position n was drawn from.
 *   draft_tokens [B, G, N-1] int32.
 *   uniforms     [B, (N-1)*G + 1] fp32 in [0,1), laid out as for
 *                sv_verify_lookahead_sample.
 *   B >= 0, 1 <= G <= 32, N >= 2, G*N <= 1024, G*G*(N-1) <= 2048, V >= 2;
 *   B*G*(2N-1) < 2^31; temperature > 0 (finite), on both sides.
 * Draft g's token x is accepted when u < min(1, p(x)/q_g(x)) (q_g(x) = 0 <
 * p(x) accepts, p(x) = 0 rejects), p the current distribution; a rejection
 * replaces p by norm(max(0, p - q_g)) (p itself if that is all zero).
 * Outputs as for sv_verify_lookahead_sample; out_row_lse, if given, holds
 * B*G*N target rows then B*G*(N-1) draft rows. Bad input also covers every
 * draft row.
 */
int sv_verify_multidraft_sample(const void* target, const void* draft, const int32_t* draft_tokens,
                                const float* uniforms, int64_t B, int32_t G, int32_t N, int64_t V, int32_t dtype,
                                float temperature, int32_t* out_tokens, int32_t* out_accept_len,
                                int32_t* out_best_cand, float* out_row_lse, void* stream);

/*
 * Sampling-mode verify on hidden states: the target's and the draft's logits
 * are computed here from their last hidden states and LM heads, on the
 * tensor cores, then verified exactly as sv_verify_sample verifies logits.
 * The pages take the logits as given ("Speculative Decoding —— LLM推理优化技术
 * （一）" §2.1-2.3, §4: p = softmax(target logits / T), q likewise); this entry
 * point produces them as logits = h · Wᵀ.
 *
 *   h_target [B, K+1, D] bf16, h_draft [B, K, D] bf16: the hidden states at
 *            the positions whose logits sv_verify_sample would take.
 *   w_target, w_draft [V, D] bf16: the two LM heads (row v is vocabulary
 *            entry v).
 *   D a multiple of 64, below 2^31; B*(2K+1) < 2^31; the four arrays
 *            16-byte aligned.
 *   draft_tokens, uniforms, B, K, V, temperature (> 0), top_p, out_tokens,
 *   out_accept_len: as for sv_verify_sample.
 *   out_logits nullable [B*(K+1) + B*K, V] fp32: where to put the logits
 *            (target rows, then draft rows); without it the library keeps a
 *            workspace per (device, stream), freed by sv_release().
 * The products of bf16 values are exact in fp32 and the sums are fp32: the
 * logits equal h · Wᵀ up to fp32 summation rounding. On `stream`: the GEMM
 * (its operands read by tensor copies), then the kernels sv_verify_sample
 * runs on fp32 logits of this shape. SV_ERR_CUDA also when the driver offers
 * no tensor-map encoder.
 */
int sv_verify_sample_lmhead(const void* h_target, const void* h_draft, const void* w_target, const void* w_draft,
                            const int32_t* draft_tokens, const float* uniforms, int64_t B, int32_t K, int64_t D,
                            int64_t V, float temperature, float top_p, int32_t* out_tokens, int32_t* out_accept_len,
                            float* out_logits, void* stream);

/*
 * N-gram pool of Lookahead decoding ("Lookahead Decoding 完全拆解", section
 * "N-gram 池与身份判定"; W new n-grams per step from the section on the 2D
 * window; at most G candidates, GUESS_SET_SIZE, in the engineering section).
 * The pool caches the n-grams the lookahead branch collects, one pool per
 * sequence, keyed by an n-gram's first token; only the n-grams whose first
 * token equals the sequence's last generated token are candidates for the
 * verify branch, and a lookup leaves the pool as it was (n-grams that are not
 * adopted stay). Where the page is silent this library reads: each first
 * token holds at most `cap` n-grams; a step's n-grams are inserted in order;
 * an n-gram already held is not inserted again and keeps its place;
 * inserting into a full first token drops its oldest n-gram; candidates are
 * the newest first; an n-gram with a token outside [0, V) is ignored.
 *
 * The pool lives in caller-owned device memory of sv_ngram_pool_bytes(B, V,
 * N, cap) bytes (256-byte aligned); B, V, N and cap must be the same on every
 * call that uses it. 1 <= N <= 4096 is the n-gram length (N >= 2), 1 <= cap <=
 * 4096. Calls are asynchronous on `stream` like the verify calls.
 *
 *   sv_ngram_pool_bytes: the bytes a pool needs (-1 for a bad shape).
 *   sv_ngram_pool_reset: empties the pool (a memset of its counters).
 *   sv_ngram_pool_insert: ngrams [B, W, N] int32; sequence b's W n-grams go
 *     into its pool in order.
 *   sv_ngram_pool_lookup: last [B] int32, each sequence's last generated
 *     token; writes cand [B, G, N-1] int32, the tokens after the first of the
 *     matching n-grams, newest first (the layout sv_verify_greedy reads), and
 *     count [B] int32, how many there are. Unused candidate slots hold a copy
 *     of the newest candidate, or the last token repeated when there is none
 *     (a guess that cannot change what the greedy verify outputs). A last
 *     token outside [0, V) gives count -1 and -1 tokens.
 */
int64_t sv_ngram_pool_bytes(int64_t B, int64_t V, int32_t N, int32_t cap);
int sv_ngram_pool_reset(void* pool, int64_t B, int64_t V, int32_t N, int32_t cap, void* stream);
int sv_ngram_pool_insert(void* pool, int64_t B, int64_t V, int32_t N, int32_t cap, const int32_t* ngrams,
                         int32_t W, void* stream);
int sv_ngram_pool_lookup(const void* pool, int64_t B, int64_t V, int32_t N, int32_t cap, const int32_t* last,
                         int32_t G, int32_t* cand, int32_t* count, void* stream);

/*
 * sv_verify_sample_noalloc: sv_verify_sample for callers that cannot allocate
 * device memory. The pages have no counterpart to this entry point; it exists
 * for deployment constraints, not for the method.
 *
 * Who needs it: code that runs inside a caller-managed memory pool or arena
 * that must account for every byte, allocator hooks that would recurse into
 * themselves if the library called cudaMalloc, and services that reserve all
 * device memory at start-up and treat any later allocation as a failure.
 * sv_verify_sample allocates a scratch area per stream on its first call; this
 * entry point never allocates: it uses a fixed 4 MiB scratch array that is
 * part of the library image and that every GPU which loads the library holds
 * until the process exits.
 *
 * Arguments, outputs and results are exactly those of sv_verify_sample: the
 * same argument checks, the same choice of kernels and the same launch
 * shapes; only the scratch differs. Differences:
 *   - A call whose scratch would exceed 4 MiB returns SV_ERR_SCRATCH_LIMIT and
 *     enqueues nothing. On the row pass + decide kernels (see
 *     sv_set_sample_path) the scratch is 512 + 8*B*R*NCH + 8*B*K + 48*B bytes,
 *     each term rounded up to 256, with R = 2K+1 rows per sequence and
 *     NCH = ceil(V*s/32768) chunks per row (s = 2 for bf16, 4 for fp32; 1 when
 *     a row holds at most 16 KB); with top-p the 8*B*R*NCH term is 16*B*R.
 *     E.g. about 0.3 MiB for B=256, K=8, V=128256 bf16. On the streaming
 *     kernel it is about 256 + 4*(B*R + B*(3+D)) + 8*B*R*ceil(NT/CT) +
 *     16*B*R + 48*B bytes, plus 4*B*ceil(V/256) when the draws are split over
 *     D > 0 chunks.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, with the device current) and caches it;
 *     make that first call before any stream capture.
 *   - Each call clears the array's control block and counters with a memset
 *     on `stream` before its kernel.
 *   - All calls on all streams share the one array, which keeps the contents
 *     the last call left. Calls whose kernels overlap on the GPU race on it:
 *     issue them on one stream, or otherwise keep them from overlapping.
 *   - sv_get_status() does not report this entry point's device-side input
 *     errors; out_accept_len[b] == -1 still marks a sequence with bad input.
 */
int sv_verify_sample_noalloc(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                             const float* uniforms, int64_t B, int32_t K, int64_t V, int32_t dtype, float temperature,
                             float top_p, int32_t* out_tokens, int32_t* out_accept_len, float* out_row_stats,
                             void* stream);

/*
 * Synchronises `stream`, then returns and clears the sticky device status of
 * that stream's scratch: SV_OK, SV_ERR_INPUT (some sequence had bad input
 * since the last call) or SV_ERR_TIMEOUT (a bounded wait ran out; the scratch
 * has been re-zeroed so later calls start clean). SV_ERR_CUDA if the
 * synchronisation itself failed.
 */
int sv_get_status(void* stream);

/*
 * Self-test of the failure path (the pages have no counterpart; it exists so
 * that the timeout handling can be tested without any fault): enqueues on
 * `stream` a one-thread kernel that waits for a control word nothing ever
 * sets, gives up after limit_ns nanoseconds (0..2e9) exactly as every
 * internal wait does, and records SV_ERR_TIMEOUT in the stream's status. A
 * following sv_get_status(stream) returns SV_ERR_TIMEOUT and resets the
 * stream's scratch; later calls work as before. Returns SV_ERR_ARG for a
 * limit outside the range, SV_ERR_NOMEM / SV_ERR_CUDA as the other calls.
 */
int sv_selftest_wait_timeout(int64_t limit_ns, void* stream);

/* Synchronises `stream` and returns how many sampling draws on that stream's
 * scratch area were redone in double-float arithmetic so far (the fp32 walk
 * found u*Z within 1e-7*Z of an edge of the token's CDF interval); -1 on a
 * CUDA error. For monitoring; the pages have no counterpart. */
int64_t sv_refined_draws(void* stream);

/* A static, human-readable name for an sv_status value. */
const char* sv_status_string(int status);

/* Frees every scratch area on every device (synchronises those devices). */
int sv_release(void);

/* Launch-shape knobs, for tuning and tests: stages of the shared-memory ring
 * (1..6) and CTAs per SM (1..4); 0 restores the default. Applies to calls
 * made after it on any device. */
int sv_set_launch_shape(int32_t stages, int32_t ctas_per_sm);

/* How many kernel launches the library has enqueued since it was loaded. */
uint64_t sv_launch_count(void);

/* Which kernels sv_verify_greedy uses, for comparing them: 0 (default) one
 * CTA per row for the argmax, then one warp per sequence for the match; 1 the
 * streaming kernel. Applies to calls made after it. */
int sv_set_greedy_path(int32_t path);

/* Which kernels sv_verify_sample uses, for comparing them. 0 (default):
 * with T > 0 and top_p = 1, rows of at most 1024 elements go to the
 * streaming kernel's one-warp-per-sequence mode; calls whose logits are at
 * most 96 MiB (so that the second look at the draw rows hits L2) to the row
 * pass and the cluster decide kernel; with top_p < 1, bf16 rows with V a
 * multiple of 8 and V <= 327680 (16-byte aligned logits, K <= 1024) go to
 * the row pass in its top-p form (one thread-block cluster per row) and the
 * decide kernel at every size; everything else (larger calls, other top-p
 * calls, T = 0) to the streaming kernel. 1: always the streaming kernel,
 * including its sequence-in-shared-memory mode (whose draws are not handed
 * to the refine kernel). 2: the row pass and decide kernel wherever they fit
 * (top_p = 1: T > 0, K <= 1024, V <= 1048576; top_p < 1 as for 0). Applies
 * to calls made after it. */
int sv_set_sample_path(int32_t path);

#ifdef __cplusplus
}
#endif
#endif
