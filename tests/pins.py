"""Checks that pin the CPU oracle to what the pages and the mathematics fix.

Each check takes the oracle library to test (``lib``), so the same check can be
run against the real oracle and against builds with a planted mistake
(tests/test_oracle_mutations.py), which it must reject.

Sources (page title, section):
  "Speculative Decoding —— LLM推理优化技术（一）" (hustzhy.cn), §2.2: the output
      follows p; §2.4: E[accept] = 1 - TV(p, q); §3.1: tokens per round
      (1 - a^(K+1)) / (1 - a).
  "Lookahead Decoding 完全拆解" (pinghaoyang.com.cn), scaling-law section,
      eq. (5): E[#tokens] = (g+1) - sum_{i=1..g} (1 - a^i)^b for b drafts;
      section "采样模式的验证": greedily produced candidates have a one-hot
      draft distribution, and the sampling-mode verify keeps the target's
      output distribution.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
from scipy import stats

import oracle
import specgen as sg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def softmax(l, T=1.0):
    z = np.asarray(l, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def nucleus_bruteforce(l, p, top_p):
    """The largest threshold whose upper set holds >= top_p (all distinct values tried)."""
    l = np.asarray(l, np.float64)
    for tau in sorted(set(l.tolist()), reverse=True):
        if p[l >= tau].sum() >= top_p:
            return tau
    return l.min()


def dist(l, T, top_p=1.0):
    p = softmax(l, T)
    if top_p < 1:
        tau = nucleus_bruteforce(l, p, top_p)
        p = np.where(np.asarray(l) >= tau, p, 0.0)
        p /= p.sum()
    return p


def replicate(target_rows, draft_rows, n):
    t = np.broadcast_to(np.asarray(target_rows, np.float32), (n,) + np.shape(target_rows)).copy()
    d = np.broadcast_to(np.asarray(draft_rows, np.float32), (n,) + np.shape(draft_rows)).copy()
    return t, d


# Fixed small rows used by the statistical checks (V = 8).
LT = np.array([[1.0, 0.5, -0.3, 2.0, 0.0, -1.0, 1.5, 0.2],
               [0.3, 1.7, -0.5, 0.1, 1.1, -2.0, 0.4, 0.9]], np.float32)
LD = np.array([[0.2, 1.1, 0.4, 1.2, 0.9, -0.2, 0.3, 1.0]], np.float32)


def check_output_is_target_distribution(lib, T=1.0, top_p=1.0, n=1_000_000, seed=11):
    """§2.2: the emitted token at position 0 follows p_0 (chi-square, df = V-1);
    given all K=1 draft tokens accepted, the bonus follows p_1."""
    V = LT.shape[1]
    target, draft = replicate(LT, LD, n)
    toks = sg.draft_tokens(draft, sg.F32, T, top_p, seed=seed)
    u = sg.uniforms(n, 1, seed=seed)
    out, acc, _ = oracle.verify_sample(target, draft, toks, u, T, top_p, lib=lib)
    assert (acc >= 0).all()
    for pos, rows in ((0, np.ones(n, bool)), (1, acc == 1)):
        p = dist(LT[pos], T, top_p)
        c = np.bincount(out[rows, pos], minlength=V)
        keep = p > 0
        assert c[~keep].sum() == 0, "emitted a token outside the target's support"
        _, pval = stats.chisquare(c[keep], p[keep] * rows.sum())
        assert pval > 1e-3, f"position {pos}: chi-square p-value {pval:.3g}"


def check_acceptance_is_one_minus_tv(lib, T=1.0, n=1_000_000, seed=12):
    """§2.4: P(accept x_0) = sum_x min(p, q) = 1 - TV(p, q), within 4 sigma."""
    target, draft = replicate(LT, LD, n)
    toks = sg.draft_tokens(draft, sg.F32, T, 1.0, seed=seed)
    u = sg.uniforms(n, 1, seed=seed)
    _, acc, _ = oracle.verify_sample(target, draft, toks, u, T, 1.0, lib=lib)
    p, q = softmax(LT[0], T), softmax(LD[0], T)
    alpha = np.minimum(p, q).sum()
    assert abs(alpha - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
    rate = (acc == 1).mean()
    assert abs(rate - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / n), (rate, alpha)


def check_tokens_per_round(lib, K, n=200_000, seed=13):
    """§3.1: with the same (p, q) at every position, acceptances are iid with
    rate a and E[tokens per round] = (1 - a^(K+1)) / (1 - a)."""
    lt = LT[0]
    ld = LD[0]
    target, draft = replicate(np.tile(lt, (K + 1, 1)), np.tile(ld, (K, 1)), n)
    toks = sg.draft_tokens(draft, sg.F32, 1.0, 1.0, seed=seed + K)
    u = sg.uniforms(n, K, seed=seed + K)
    _, acc, _ = oracle.verify_sample(target, draft, toks, u, 1.0, 1.0, lib=lib)
    a = np.minimum(softmax(lt), softmax(ld)).sum()
    expect = (1 - a ** (K + 1)) / (1 - a)
    tokens = acc + 1.0
    assert abs(tokens.mean() - expect) < 4 * tokens.std() / math.sqrt(n), (tokens.mean(), expect)


# Distributions whose probabilities are multiples of 1/8, so that every accept
# threshold and every CDF edge is a multiple of 1/16 and a midpoint grid of
# uniforms integrates the oracle's decisions exactly.
NICE_P = [np.array([3, 3, 1, 1]) / 8, np.array([1, 2, 4, 1]) / 8, np.array([1, 1, 2, 4]) / 8]
NICE_Q = [np.array([2, 2, 2, 2]) / 8, np.array([2, 1, 1, 4]) / 8]


def closed_form_mass(K, j, t):
    """§2.2-2.3: P(output = t_0..t_j with accept length j)
    = prod_{i<j} min(p_i, q_i)(t_i) * (max(0, p_j - q_j)(t_j) if j < K else p_K(t_K))."""
    m = 1.0
    for i in range(j):
        m *= min(NICE_P[i][t[i]], NICE_Q[i][t[i]])
    if j < K:
        m *= max(0.0, NICE_P[j][t[j]] - NICE_Q[j][t[j]])
    else:
        m *= NICE_P[K][t[K]]
    return m


def check_brute_force(lib, K=2, n=16):
    """Enumerate every draft tuple (weight prod q_i(x_i)) and a midpoint grid
    of n^(K+1) uniform vectors; the mass of each output equals the closed form."""
    V = 4
    lt = np.log(np.array(NICE_P[: K] + [NICE_P[K]]))
    ld = np.log(np.array(NICE_Q[:K]))
    grid = (np.arange(n) + 0.5) / n
    U = np.array(list(itertools.product(grid, repeat=K + 1)), np.float32)
    B = U.shape[0]
    target, draft = replicate(lt, ld, B)
    mass = {}
    for x in itertools.product(range(V), repeat=K):
        w = np.prod([NICE_Q[i][x[i]] for i in range(K)])
        if w == 0:
            continue
        toks = np.tile(np.array(x, np.int32), (B, 1))
        out, acc, _ = oracle.verify_sample(target, draft, toks, U, 1.0, 1.0, lib=lib)
        assert (acc >= 0).all()
        keys, counts = np.unique(np.concatenate([acc[:, None], out], 1), axis=0, return_counts=True)
        for k, c in zip(keys, counts):
            key = (int(k[0]),) + tuple(int(v) for v in k[1: 2 + k[0]])
            mass[key] = mass.get(key, 0.0) + w * c / B
    total = 0.0
    for j in range(K + 1):
        for t in itertools.product(range(V), repeat=j + 1):
            expect = closed_form_mass(K, j, t)
            got = mass.get((j,) + t, 0.0)
            assert abs(got - expect) < 1e-9, ((j,) + t, got, expect)
            total += expect
    assert abs(total - 1.0) < 1e-12
    assert abs(sum(mass.values()) - 1.0) < 1e-9


def check_draw_edge_rules(lib):
    """The draw's two edge rules, on hand-made weights (readings c5 and c7).

    c5 ("Speculative Decoding" §2.1 inverse CDF, ascending vocabulary order,
    strict comparison): the smallest t with C_t > u*Z; when u*Z is at or past
    the last partial sum (here u = 1, which a valid uniform never is), the
    largest t with positive weight. c7 ("Speculative Decoding" §4, the
    fallback when the residual sums to zero): with p <= q everywhere the
    residual max(0, p - q) is all zero and the token is drawn from p itself.
    Expected tokens are worked out by hand in the comments."""
    w = np.array([0.5, 0.25, 0.25, 0.0, 0.0])
    # u*Z = 0.5: C_0 = 0.5 is not > 0.5, C_1 = 0.75 is -> token 1
    assert oracle.inverse_cdf(w, 0.5, lib) == 1
    # u = 0: the first token with positive weight
    assert oracle.inverse_cdf(np.array([0.0, 0.0, 1.0, 0.0]), 0.0, lib) == 2
    # u*Z = Z: no partial sum exceeds it -> the largest t with w_t > 0 (2, not V-1)
    assert oracle.inverse_cdf(w, 1.0, lib) == 2
    assert oracle.inverse_cdf(np.array([0.0, 0.0, 1.0, 0.0]), 1.0, lib) == 2
    # residual max(0, p - q) = [0, 0.4, 0]: every u draws token 1
    p, q = np.array([0.1, 0.6, 0.3]), np.array([0.4, 0.2, 0.4])
    for u in (0.0, 0.3, 0.99):
        assert oracle.residual_draw(p, q, u, lib) == 1
    # p <= q everywhere: the residual is zero, the draw is from p: u*Z = 0.5 < C_0 = 0.6 -> 0
    # (from q it would be 0.9 -> 1; from max(0, q - p) = [0, .4, .4] it would be 2)
    p, q = np.array([0.6, 0.2, 0.2]), np.array([0.6, 0.6, 0.6])
    assert oracle.residual_draw(p, q, 0.5, lib) == 0
    # from p, u*Z = 0.85: C = 0.6, 0.8, 1.0 -> 2
    assert oracle.residual_draw(p, q, 0.85, lib) == 2


def load_topp_golden():
    cases = []
    for line in open(os.path.join(GOLDEN, "topp_ties.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        head, logits, kept, ps, tau = [s.strip() for s in line.split(";")]
        T, top_p = (float(x) for x in head.split())
        cases.append((T, top_p, np.array(logits.split(), np.float32), [int(k) for k in kept.split()],
                      float(ps), float(tau)))
    return cases


def check_topp_golden(lib):
    for T, top_p, l, kept, ps, tau in load_topp_golden():
        st = oracle.row_stats(l[None, :], T, top_p, lib=lib)[0]
        assert abs(st[2] - ps) < 2e-6, (T, top_p, st, ps)
        assert st[3] == tau, (T, top_p, st, tau)
        assert sorted(np.nonzero(l >= st[3])[0].tolist()) == kept


def load_greedy_golden():
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "greedy_hand.txt")) if l.strip() and l[0] != "#"]
    cases, i = [], 0
    while i < len(lines):
        _, G, N, V = lines[i].split()
        G, N, V = int(G), int(N), int(V)
        rows = [[float(x) for x in lines[i + 1 + r].split()] for r in range(G * N)]
        cand = [[int(x) for x in lines[i + 1 + G * N + g].split()] for g in range(G)]
        exp = lines[i + 1 + G * N + G]
        toks, acc, best = [s.strip() for s in exp[len("expect"):].split(";")]
        cases.append((np.array(rows, np.float32).reshape(1, G, N, V), np.array(cand, np.int32).reshape(1, G, N - 1),
                      [int(t) for t in toks.split()], int(acc), int(best)))
        i += 2 + G * N + G
    return cases


def check_greedy_golden(lib):
    for logits, cand, toks, acc, best in load_greedy_golden():
        for dt in (sg.F32, sg.BF16):
            out, a, b = oracle.verify_greedy(sg.from_float(logits, dt), cand, lib=lib)
            assert out[0].tolist() == toks and a[0] == acc and b[0] == best, (out, a, b, toks, acc, best)


def multi_draft_expected_tokens(gamma, b, a, r=0.0):
    """Lookahead eq. (5) generalised to chance matches: a candidate token is the
    argmax with probability a per step until the first miss; a missed or later
    token is a uniform id that still equals the argmax with probability r.
    With r = 0 this is (g+1) - sum_i (1 - a^i)^b."""
    e = 1.0
    for i in range(1, gamma + 1):
        p_match = a ** i + sum(a ** k * (1 - a) * r ** (i - k) for k in range(i))
        e += 1.0 - (1.0 - p_match) ** b
    return e


def check_greedy_multi_draft(lib, V=512, B=12_000):
    cfg = sg.CONFIGS["cfg4_greedy_v32000_bf16"].with_(B=B, V=V, seed=5)
    d = sg.greedy_inputs(cfg)
    _, acc, _ = oracle.verify_greedy(d["logits"], d["cand"], lib=lib)
    assert (acc >= 0).all()
    tokens = acc + 1.0
    expect = multi_draft_expected_tokens(cfg.N - 1, cfg.G, cfg.match_prob, 1.0 / V)
    assert abs(tokens.mean() - expect) < 4 * tokens.std() / math.sqrt(B), (tokens.mean(), expect)


# ---------------------------------------------------------------------------
# Lookahead sampling-mode verify ("Lookahead Decoding 完全拆解", section
# "采样模式的验证"): candidates come from greedy decoding, so each one's draft
# distribution is one-hot on its token; the verify only decides acceptance and
# leaves the target distribution intact.

def lookahead_law(P, cand):
    """Law of the verify's output, from the page's invariance claim alone.

    P[g][n] is the target distribution at position n of candidate g's branch,
    cand[g][n] its token (n < N-1). Every emitted token follows the target:
    position n's token t is drawn from P[lead][n], where lead owns the accepted
    prefix (candidate 0 at n = 0). t extends the prefix when a candidate still
    matching the prefix holds t at n (the new owner is the lowest such
    candidate); otherwise the round ends with t. Row N-1 gives the bonus.
    Returns {(accept_len, t_0, .., t_j): probability}."""
    G, N = len(P), len(P[0])
    V = len(P[0][0])
    law = {}

    def walk(n, alive, lead, prefix, mass):
        p = P[lead][n]
        if n == N - 1:
            for t in range(V):
                if p[t]:
                    law[(n,) + prefix + (t,)] = law.get((n,) + prefix + (t,), 0) + mass * p[t]
            return
        held = {cand[g][n] for g in alive}
        for t in range(V):
            if not p[t]:
                continue
            if t in held:
                nxt = [g for g in alive if cand[g][n] == t]
                walk(n + 1, nxt, min(nxt), prefix + (t,), mass * p[t])
            else:
                law[(n,) + prefix + (t,)] = law.get((n,) + prefix + (t,), 0) + mass * p[t]

    walk(0, list(range(G)), 0, (), 1)
    return law


def lookahead_outcomes(out, acc):
    """Tally (accept_len, t_0..t_j) keys of a batch of verify outputs."""
    keys = np.concatenate([acc[:, None], out], 1)
    uniq, counts = np.unique(keys, axis=0, return_counts=True)
    res = {}
    for k, c in zip(uniq, counts):
        res[(int(k[0]),) + tuple(int(v) for v in k[1: 2 + k[0]])] = int(c)
    return res


F = __import__("fractions").Fraction
# Two shapes with G = 2, N = 3, V = 4 whose probabilities are multiples of
# 1/12 and are picked so that every accept threshold and every CDF edge the
# walk can meet (after removing rejected tokens and renormalising) is again a
# multiple of 1/12: a midpoint grid of 12 values per uniform then integrates
# the oracle's decisions exactly. Shape "shared": both candidates start with
# the same token. Shape "split": they differ from the first token on.
LA_EXACT = {
    "shared": ([[[F(6, 12), F(3, 12), F(2, 12), F(1, 12)], [F(6, 12), F(2, 12), F(3, 12), F(1, 12)],
                 [F(3, 12)] * 4],
                [[F(1, 12), F(2, 12), F(3, 12), F(6, 12)], [F(2, 12), F(4, 12), F(3, 12), F(3, 12)],
                 [F(6, 12), F(2, 12), F(2, 12), F(2, 12)]]],
               [[0, 0], [0, 2]]),
    "split": ([[[F(6, 12), F(3, 12), F(2, 12), F(1, 12)], [F(6, 12), F(2, 12), F(3, 12), F(1, 12)],
                [F(3, 12)] * 4],
               [[F(1, 12), F(2, 12), F(3, 12), F(6, 12)], [F(2, 12), F(6, 12), F(2, 12), F(2, 12)],
                [F(6, 12), F(2, 12), F(2, 12), F(2, 12)]]],
              [[0, 0], [1, 1]]),
}


def check_lookahead_exact(lib, shape, dtype=sg.F32, n=12):
    """Every output's mass, integrated over the n^5 midpoint grid of uniforms,
    equals lookahead_law exactly (up to the rounding of ln p in storage)."""
    P, cand = LA_EXACT[shape]
    G, N, V = len(P), len(P[0]), len(P[0][0])
    logits = np.log(np.array([[[float(x) for x in row] for row in rows] for rows in P]))
    grid = (np.arange(n) + 0.5) / n
    U = np.array(list(itertools.product(grid, repeat=(N - 1) * G + 1)), np.float32)
    B = U.shape[0]
    L = np.broadcast_to(sg.from_float(logits, dtype), (B, G, N, V)).copy()
    C = np.broadcast_to(np.array(cand, np.int32), (B, G, N - 1)).copy()
    out, acc, best, _ = oracle.verify_lookahead_sample(L, C, U, 1.0, lib=lib)
    assert (acc >= 0).all()
    got = lookahead_outcomes(out, acc)
    law = lookahead_law(P, cand)
    assert sum(law.values()) == 1
    for key in set(got) | set(law):
        assert abs(got.get(key, 0) / B - float(law.get(key, 0))) < 1e-9, (shape, key, got.get(key, 0) / B,
                                                                          law.get(key, 0))


LA_CAND = [[2, 0], [2, 3], [4, 0]]  # G = 3, N = 3: a shared first token, a split, a repeat


def check_lookahead_chisquare(lib, T=0.8, n=400_000, seed=21):
    """The output law of random rows (V = 5, G = 3, N = 3) against
    lookahead_law by chi-square over every outcome (small ones pooled)."""
    G, N, V = 3, 3, 5
    rows = np.random.default_rng(seed).normal(0, 1.2, size=(G, N, V)).astype(np.float32)
    P = [[softmax(rows[g, k], T).tolist() for k in range(N)] for g in range(G)]
    law = lookahead_law(P, LA_CAND)
    L = np.broadcast_to(rows, (n, G, N, V)).copy()
    C = np.broadcast_to(np.array(LA_CAND, np.int32), (n, G, N - 1)).copy()
    U = sg.uniforms(n, (N - 1) * G, seed=seed)
    out, acc, _, _ = oracle.verify_lookahead_sample(L, C, U, T, lib=lib)
    got = lookahead_outcomes(out, acc)
    assert set(got) <= set(law), "an outcome the law gives probability zero"
    keys = sorted(law, key=lambda k: -law[k])
    exp = np.array([law[k] * n for k in keys])
    obs = np.array([got.get(k, 0) for k in keys], float)
    big = exp >= 20
    exp = np.append(exp[big], exp[~big].sum())
    obs = np.append(obs[big], obs[~big].sum())
    _, pval = stats.chisquare(obs, exp)
    assert pval > 1e-3, f"chi-square p-value {pval:.3g}"


def check_lookahead_single_candidate(lib, seed=22):
    """G = 1 is the sampling-mode verify with a one-hot draft row (logit 0 on
    the candidate, -inf elsewhere); candidates all equal to candidate 0 give
    the same result as candidate 0 alone (a repeated token is already removed)."""
    B, N, V, T = 3000, 5, 16, 0.9
    rng = np.random.default_rng(seed)
    rows = sg.from_float(rng.normal(0, 1.5, size=(B, 1, N, V)), sg.F32)
    cand = rng.integers(0, V, size=(B, 1, N - 1)).astype(np.int32)
    U = sg.uniforms(B, N - 1, seed=seed)
    draft = np.full((B, N - 1, V), -np.inf, np.float32)
    np.put_along_axis(draft, cand[:, 0, :, None], 0.0, axis=2)
    out_s, acc_s, _ = oracle.verify_sample(rows[:, 0], draft, cand[:, 0], U, T, lib=lib)
    out_l, acc_l, best, _ = oracle.verify_lookahead_sample(rows, cand, U, T, lib=lib)
    assert (acc_s >= 0).all() and (best == 0).all()
    np.testing.assert_array_equal(acc_l, acc_s)
    np.testing.assert_array_equal(out_l, out_s)
    G = 3
    rows3 = np.repeat(rows, G, axis=1)
    cand3 = np.repeat(cand, G, axis=1)
    U3 = np.zeros((B, (N - 1) * G + 1), np.float32)
    for k in range(N - 1):
        U3[:, k * G] = U[:, k]
        U3[:, k * G + 1: (k + 1) * G] = sg.uniforms(B, G - 2, seed=seed + 1 + k)
    U3[:, -1] = U[:, -1]
    out3, acc3, best3, _ = oracle.verify_lookahead_sample(rows3, cand3, U3, T, lib=lib)
    np.testing.assert_array_equal(acc3, acc_s)
    np.testing.assert_array_equal(out3, out_s)
    assert (best3 == 0).all()


def load_lookahead_golden():
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "lookahead_sample_hand.txt"))
             if l.strip() and l[0] != "#"]
    cases, i = [], 0
    while i < len(lines):
        _, G, N, V, T = lines[i].split()
        G, N, V, T = int(G), int(N), int(V), float(T)
        rows = [[float(x) for x in lines[i + 1 + r].split()] for r in range(G * N)]
        cand = [[int(x) for x in lines[i + 1 + G * N + g].split()] for g in range(G)]
        u = [float(x) for x in lines[i + 1 + G * N + G].split()[1:]]
        exp = lines[i + 2 + G * N + G]
        toks, acc, best = [s.strip() for s in exp[len("expect"):].split(";")]
        cases.append((np.array(rows, np.float32).reshape(1, G, N, V), np.array(cand, np.int32).reshape(1, G, N - 1),
                      np.array(u, np.float32).reshape(1, -1), T, [int(t) for t in toks.split()], int(acc),
                      int(best)))
        i += 3 + G * N + G
    return cases


def check_lookahead_golden(lib):
    for logits, cand, u, T, toks, acc, best in load_lookahead_golden():
        out, a, b, _ = oracle.verify_lookahead_sample(logits, cand, u, T, lib=lib)
        assert out[0].tolist() == toks and a[0] == acc and b[0] == best, (out, a, b, toks, acc, best)


# ---------------------------------------------------------------------------
# Multi-draft sampling verify: G drafts, each drawn from its own draft
# distribution, verified by the walk above with alpha = min(1, p(x)/q_g(x)) and
# the residual norm(max(0, p - q_g)) after each rejection ("Speculative
# Decoding —— LLM推理优化技术（一）" §2.1-2.2, applied once per rejected draft).

def one_hot_rows(tokens, V):
    """Draft logits that put all mass on the given tokens: 0 there, -inf elsewhere."""
    rows = np.full(tokens.shape + (V,), -np.inf, np.float32)
    np.put_along_axis(rows, tokens[..., None], 0.0, axis=-1)
    return rows


def check_multidraft_one_hot_is_lookahead(lib, seed=31):
    """One-hot draft rows make the multi-draft verify the Lookahead one."""
    B, G, N, V, T = 2000, 4, 4, 12, 0.8
    rng = np.random.default_rng(seed)
    target = rng.normal(0, 1.5, size=(B, G, N, V)).astype(np.float32)
    cand = rng.integers(0, 3, size=(B, G, N - 1)).astype(np.int32)  # few distinct tokens: shared prefixes
    U = sg.uniforms(B, (N - 1) * G, seed=seed)
    m = oracle.verify_multidraft_sample(target, one_hot_rows(cand, V), cand, U, T, lib=lib)
    la = oracle.verify_lookahead_sample(target, cand, U, T)
    for a, b in zip(m[:3], la[:3]):
        np.testing.assert_array_equal(a, b)


def check_multidraft_single_draft_is_sampling(lib, seed=32):
    """One draft makes it the sampling-mode verify with K = N-1."""
    B, N, V, T = 3000, 5, 10, 0.9
    rng = np.random.default_rng(seed)
    target = rng.normal(0, 1.5, size=(B, 1, N, V)).astype(np.float32)
    draft = (target[:, :, : N - 1] + rng.normal(0, 1.0, size=(B, 1, N - 1, V))).astype(np.float32)
    toks = sg.draft_tokens(draft[:, 0], sg.F32, T, 1.0, seed=seed)
    U = sg.uniforms(B, N - 1, seed=seed)
    out, acc, best, _ = oracle.verify_multidraft_sample(target, draft, toks[:, None, :], U, T, lib=lib)
    rt, ra, margin = oracle.verify_sample(target[:, 0], draft[:, 0], toks, U, T)
    assert (best == 0).all() and (ra >= 0).all()
    firm = margin > 1e-9  # the two normalise the residual in a different order
    np.testing.assert_array_equal(acc[firm], ra[firm])
    np.testing.assert_array_equal(out[firm], rt[firm])


MD_G, MD_N, MD_V = 3, 3, 6


def multidraft_case(n, T, seed):
    """Fixed target and draft rows (draft g's rows near the target's, so that
    drafts are often accepted), drafts sampled from their own rows."""
    rng = np.random.default_rng(seed)
    lt = rng.normal(0, 1.0, size=(MD_G, MD_N, MD_V)).astype(np.float32)
    ld = (lt[:, : MD_N - 1] + rng.normal(0, 0.8, size=(MD_G, MD_N - 1, MD_V))).astype(np.float32)
    target = np.broadcast_to(lt, (n,) + lt.shape).copy()
    draft = np.broadcast_to(ld, (n,) + ld.shape).copy()
    toks = sg.draft_tokens(draft.reshape(n * MD_G, MD_N - 1, MD_V), sg.F32, T, 1.0, seed=seed)
    toks = toks.reshape(n, MD_G, MD_N - 1)
    U = sg.uniforms(n, (MD_N - 1) * MD_G, seed=seed + 1)
    return lt, target, draft, toks, U


def check_multidraft_marginal(lib, T=0.9, n=300_000, seed=33):
    """Over drafts drawn from their rows, the first token follows the target
    row of candidate 0; given an accepted first token t_0, the next token
    follows the target row of the lowest draft starting with t_0 (chi-square).
    The accepted prefix is the reported owner's, and no lower draft has it."""
    lt, target, draft, toks, U = multidraft_case(n, T, seed)
    out, acc, best, _ = oracle.verify_multidraft_sample(target, draft, toks, U, T, lib=lib)
    assert (acc >= 0).all()
    for b in np.nonzero(acc >= 1)[0][:20000]:
        j, g = acc[b], best[b]
        assert (out[b, :j] == toks[b, g, :j]).all()
        assert not any((toks[b, h, :j] == out[b, :j]).all() for h in range(g))
    p0 = softmax(lt[0, 0], T)
    _, pval = stats.chisquare(np.bincount(out[:, 0], minlength=MD_V), p0 * n)
    assert pval > 1e-3, f"position 0: chi-square p-value {pval:.3g}"
    ext = acc >= 1
    owner = np.argmax(toks[:, :, 0] == out[:, 0:1], axis=1)  # lowest draft holding t_0
    for a in range(MD_G):
        rows = ext & (owner == a)
        if rows.sum() < 2000:
            continue
        p1 = softmax(lt[a, 1], T)
        _, pval = stats.chisquare(np.bincount(out[rows, 1], minlength=MD_V), p1 * rows.sum())
        assert pval > 1e-3, f"position 1 after owner {a}: chi-square p-value {pval:.3g}"


def load_multidraft_golden():
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "multidraft_sample_hand.txt"))
             if l.strip() and l[0] != "#"]
    cases, i = [], 0
    while i < len(lines):
        _, G, N, V, T = lines[i].split()
        G, N, V, T = int(G), int(N), int(V), float(T)
        k = i + 1
        tgt = [[float(x) for x in lines[k + r].split()] for r in range(G * N)]
        k += G * N
        dft = [[float(x) for x in lines[k + r].split()] for r in range(G * (N - 1))]
        k += G * (N - 1)
        toks = [[int(x) for x in lines[k + g].split()] for g in range(G)]
        k += G
        u = [float(x) for x in lines[k].split()[1:]]
        exp = lines[k + 1]
        out, acc, best = [s.strip() for s in exp[len("expect"):].split(";")]
        cases.append((np.array(tgt, np.float32).reshape(1, G, N, V), np.array(dft, np.float32).reshape(1, G, N - 1, V),
                      np.array(toks, np.int32).reshape(1, G, N - 1), np.array(u, np.float32).reshape(1, -1), T,
                      [int(t) for t in out.split()], int(acc), int(best)))
        i = k + 2
    return cases


def check_multidraft_golden(lib):
    for tgt, dft, toks, u, T, out_e, acc_e, best_e in load_multidraft_golden():
        out, acc, best, _ = oracle.verify_multidraft_sample(tgt, dft, toks, u, T, lib=lib)
        assert out[0].tolist() == out_e and acc[0] == acc_e and best[0] == best_e, (out, acc, best, out_e, acc_e,
                                                                                   best_e)


# ---------------------------------------------------------------------------
# The sampling verify on logits computed by the LM heads, h · W^T (the
# computation a fused LM-head GEMM with a verify epilogue reproduces).

def check_lmhead_identity(lib, seed=41):
    """Identity heads (D = V, W = I) leave the hidden states as the logits."""
    B, K, V, T = 400, 3, 24, 0.8
    rng = np.random.default_rng(seed)
    ht = rng.normal(0, 1.5, size=(B, K + 1, V)).astype(np.float32)
    hd = (ht[:, :K] + rng.normal(0, 0.7, size=(B, K, V))).astype(np.float32)
    toks = sg.draft_tokens(hd, sg.F32, T, 1.0, seed=seed)
    U = sg.uniforms(B, K, seed=seed)
    eye = np.eye(V, dtype=np.float32)
    out, acc, _ = oracle.verify_sample_lmhead(ht, hd, eye, eye, toks, U, T, lib=lib)
    rt, ra, _ = oracle.verify_sample(ht, hd, toks, U, T)
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(out, rt)


def check_lmhead_integer_products(lib, dtype=sg.F32, seed=42):
    """With small integers in h and W every product and sum is exact, so the
    verify must see exactly numpy's h @ W.T (target head for the target rows,
    draft head for the draft rows). Square heads (D = V) so that a transposed
    head is a different, in-bounds matrix."""
    B, K, V, T = 300, 2, 12, 2.5
    D = V
    rng = np.random.default_rng(seed)
    ht = rng.integers(-3, 4, size=(B, K + 1, D)).astype(np.float32)
    hd = rng.integers(-3, 4, size=(B, K, D)).astype(np.float32)
    wt = rng.integers(-2, 3, size=(V, D)).astype(np.float32)
    wd = rng.integers(-2, 3, size=(V, D)).astype(np.float32)
    lt = (ht.astype(np.float64) @ wt.T.astype(np.float64)).astype(np.float32)
    ld = (hd.astype(np.float64) @ wd.T.astype(np.float64)).astype(np.float32)
    toks = sg.draft_tokens(ld, sg.F32, T, 1.0, seed=seed)
    U = sg.uniforms(B, K, seed=seed)
    conv = (lambda a: sg.from_float(a, sg.BF16)) if dtype == sg.BF16 else (lambda a: a)
    out, acc, _ = oracle.verify_sample_lmhead(conv(ht), conv(hd), conv(wt), conv(wd), toks, U, T, lib=lib)
    rt, ra, _ = oracle.verify_sample(lt, ld, toks, U, T)
    assert (ra >= 0).all()
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(out, rt)


def load_ngram_golden():
    """The hand-worked n-gram pool cases of tests/golden/ngram_pool_hand.txt:
    a list of (V, N, cap, G, ops), ops ("insert", [[tokens]]) or
    ("lookup", key, count, [[cand]])."""
    path = os.path.join(os.path.dirname(__file__), "golden", "ngram_pool_hand.txt")
    cases = []
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        word, rest = line.split(None, 1)
        if word == "pool":
            V, N, cap, G = (int(x) for x in rest.split())
            cases.append((V, N, cap, G, []))
        elif word == "insert":
            cases[-1][4].append(("insert", [[int(x) for x in g.split()] for g in rest.split("|")]))
        elif word == "lookup":
            left, right = rest.split("->")
            count, cands = right.split(":")
            cases[-1][4].append(("lookup", int(left), int(count),
                                 [[int(x) for x in g.split()] for g in cands.split("|")]))
    return cases


def check_ngram_golden(lib):
    """Every hand-worked insert/lookup sequence gives the expected candidates."""
    for V, N, cap, G, ops in load_ngram_golden():
        pool = oracle.NgramPool(1, V, N, cap, lib=lib)
        for op in ops:
            if op[0] == "insert":
                pool.insert(np.array([op[1]], dtype=np.int32))
            else:
                cand, count = pool.lookup(np.array([op[1]], dtype=np.int32), G)
                assert count[0] == op[2], (op, count)
                assert cand[0].tolist() == op[3], (op, cand[0].tolist())
        pool.close()


def check_ngram_properties(lib, seed=31, steps=60):
    """Properties the page fixes, on random streams of several sequences:
    every real candidate is an inserted n-gram whose first token is the key
    (the first-token filter), at most G of them, none twice; a lookup leaves
    the pool unchanged (n-grams that are not adopted stay); W new distinct
    n-grams of one key, in an empty pool that holds them, all come back,
    newest first."""
    rng = np.random.default_rng(seed)
    B, V, N, cap, G, W = 3, 12, 4, 3, 4, 5
    pool = oracle.NgramPool(B, V, N, cap, lib=lib)
    inserted = [set() for _ in range(B)]
    for _ in range(steps):
        g = rng.integers(0, V, size=(B, W, N)).astype(np.int32)
        g[:, :, 0] = rng.integers(0, 3, size=(B, W))  # few keys, so keys fill and evict
        pool.insert(g)
        for b in range(B):
            for w in range(W):
                inserted[b].add(tuple(g[b, w]))
        last = rng.integers(0, 3, size=B).astype(np.int32)
        cand, count = pool.lookup(last, G)
        cand2, count2 = pool.lookup(last, G)
        assert np.array_equal(cand, cand2) and np.array_equal(count, count2)
        for b in range(B):
            assert 0 <= count[b] <= min(G, cap)
            real = [tuple([int(last[b])] + cand[b, k].tolist()) for k in range(count[b])]
            assert len(set(real)) == len(real)
            for r in real:
                assert r in inserted[b] and r[0] == last[b]
    pool.close()
    pool = oracle.NgramPool(1, 100, 3, 8, lib=lib)
    grams = np.array([[[7, 10 + w, 20 + w] for w in range(6)]], dtype=np.int32)
    pool.insert(grams)
    cand, count = pool.lookup(np.array([7], dtype=np.int32), 8)
    assert count[0] == 6
    assert cand[0, :6].tolist() == [[10 + w, 20 + w] for w in reversed(range(6))]
    pool.close()
