"""Each pin must reject a plausible mistake: build a copy of the oracle with one
planted mistake (on the CPU, in a temporary directory) and check that at least
the named pin fails on it. The real oracle source is never modified."""
import os
import tempfile

import pytest

import oracle
from pins import (check_acceptance_is_one_minus_tv, check_brute_force, check_draw_edge_rules,
                  check_greedy_golden,
                  check_lmhead_integer_products, check_lookahead_exact, check_lookahead_golden,
                  check_multidraft_golden,
                  check_multidraft_marginal, check_ngram_golden, check_ngram_properties,
                  check_output_is_target_distribution, check_tokens_per_round)

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    # the residual is max(0, p - q), not max(0, q - p)
    "residual_sign": ("const double d = p[v] - q[v];", "const double d = q[v] - p[v];",
                      lambda lib: check_brute_force(lib, K=2)),
    # a residual that sums to zero falls back to p, not to q
    "zero_residual_from_q": ("return inverse_cdf(Z > 0.0 ? w : p, V, u, margin);",
                             "return inverse_cdf(Z > 0.0 ? w : q, V, u, margin);", check_draw_edge_rules),
    # past the last partial sum: the largest t with positive weight, not V - 1
    "past_end_last_index": ("    if (w[t] > 0.0) return t;\n  return V - 1;", "  return V - 1;",
                            check_draw_edge_rules),
    # ... and not the first positive one
    "past_end_first_positive": ("for (int64_t t = V - 1; t >= 0; --t)\n    if (w[t] > 0.0) return t;",
                                "for (int64_t t = 0; t < V; ++t)\n    if (w[t] > 0.0) return t;",
                                check_draw_edge_rules),
    # alpha = min(1, p/q), not min(1, q/p)
    "ratio_inverted": ("alpha = fmin(1.0, px / qx);", "alpha = fmin(1.0, qx / px);",
                       check_acceptance_is_one_minus_tv),
    # the residual must be renormalised (the draw compares against u * Z)
    "no_renormalise": ("double target = u * Z, C = 0.0;", "double target = u, C = 0.0;",
                       lambda lib: check_brute_force(lib, K=2)),
    # the bonus comes from target row K
    "bonus_wrong_row": ("      load_row(target, dtype, b * (K + 1) + K, V, lt);\n      row_dist(",
                        "      load_row(target, dtype, b * (K + 1) + K - 1, V, lt);\n      row_dist(",
                        lambda lib: check_brute_force(lib, K=2)),
    # draft token i is tested against target row i
    "target_row_off_by_one": ("load_row(target, dtype, b * (K + 1) + i, V, lt);\n      load_row(draft",
                              "load_row(target, dtype, b * (K + 1) + i + 1, V, lt);\n      load_row(draft",
                              lambda lib: check_brute_force(lib, K=2)),
    # the accept test uses u_i, not the sample's uniform
    "wrong_uniform": ("if ((double)u[i] < alpha) {", "if ((double)u[K] < alpha) {",
                      lambda lib: check_tokens_per_round(lib, 4)),
    # temperature on both sides
    "temperature_one_side": ("row_dist(ld, V, T, P, q, scratch, &margin);",
                             "row_dist(ld, V, 1.0, P, q, scratch, &margin);",
                             lambda lib: check_output_is_target_distribution(lib, 0.7, 1.0)),
    # top-p on both sides
    "top_p_one_side": ("row_dist(ld, V, T, P, q, scratch, &margin);",
                       "row_dist(ld, V, T, 1.0, q, scratch, &margin);",
                       lambda lib: check_output_is_target_distribution(lib, 1.0, 0.8)),
    # argmax ties go to the lowest index
    "argmax_highest_index": ("if (l[v] > l[best]) best = v;", "if (l[v] >= l[best]) best = v;",
                             check_greedy_golden),
    # equal prefix lengths: the lowest candidate wins
    "greedy_last_candidate": ("if (L > best_L) {", "if (L >= best_L) {", check_greedy_golden),
    # Lookahead sampling: a rejected candidate token leaves the distribution
    "lookahead_keeps_rejected": ("w[v] = fmax(0.0, p[v] - (v == x ? 1.0 : 0.0));", "w[v] = p[v];",
                                 lambda lib: check_lookahead_exact(lib, "shared")),
    # the distribution at position n is the row of the prefix's owner
    "lookahead_row_of_candidate_0": ("load_row(logits, dtype, (b * G + lead) * N + n, V, l);",
                                     "load_row(logits, dtype, (b * G + 0) * N + n, V, l);",
                                     lambda lib: check_lookahead_exact(lib, "split")),
    # so is the bonus row
    "lookahead_bonus_of_candidate_0": ("load_row(logits, dtype, (b * G + lead) * N + (N - 1), V, l);",
                                       "load_row(logits, dtype, (b * G + 0) * N + (N - 1), V, l);",
                                       lambda lib: check_lookahead_exact(lib, "shared")),
    # only candidates that still match the accepted prefix are tested
    "lookahead_no_prefix_filter": ("alive[g] = alive[g] && (c[g * (N - 1) + n] == x);", "alive[g] = alive[g];",
                                   lambda lib: check_lookahead_exact(lib, "split")),
    # u[n*G + g] tests candidate g at position n
    "lookahead_uniform_layout": ("if ((double)u[n * G + g] < alpha) {",
                                 "if ((double)u[g * (N - 1) + n] < alpha) {", check_lookahead_golden),
    # u = alpha rejects
    "lookahead_accept_on_equal": ("if ((double)u[n * G + g] < alpha) {", "if ((double)u[n * G + g] <= alpha) {",
                                  check_lookahead_golden),
    # the draw after a rejection uses the last uniform
    "lookahead_draw_uniform": ("out[n] = (int32_t)inverse_cdf(p, V, (double)u[(N - 1) * G], &margin);",
                               "out[n] = (int32_t)inverse_cdf(p, V, (double)u[0], &margin);",
                               check_lookahead_golden),
    # multi-draft: the residual is max(0, p - q_g)
    "multidraft_residual_sign": ("w[v] = fmax(0.0, p[v] - q[v]);", "w[v] = fmax(0.0, q[v] - p[v]);",
                                 check_multidraft_marginal),
    # alpha = min(1, p/q_g)
    "multidraft_ratio_inverted": ("alpha = fmin(1.0, px / qx);", "alpha = fmin(1.0, qx / px);",
                                  check_multidraft_marginal),
    # the residual is renormalised before the next draft's test
    "multidraft_no_renormalise": ("p[v] = w[v] / Z;", "p[v] = w[v];", check_multidraft_marginal),
    # each draft is tested against the distribution it was drawn from
    "multidraft_q_of_draft_0": ("load_row(draft, dtype, (b * G + g) * (N - 1) + n, V, l);",
                                "load_row(draft, dtype, (b * G + 0) * (N - 1) + n, V, l);", check_multidraft_golden),
    # only drafts that still match the accepted prefix are tested
    "multidraft_no_prefix_filter": ("alive[g] = alive[g] && (x[g * (N - 1) + n] == xa);", "alive[g] = alive[g];",
                                    check_multidraft_marginal),
    # the target row at position n is the owner's
    # the LM head is applied as h · W^T (W stored [V, D])
    "lmhead_transposed": ("load_logit(w_target, dtype, v * D + d)", "load_logit(w_target, dtype, d * V + v)",
                          check_lmhead_integer_products),
    # the draft rows use the draft model's head
    "lmhead_draft_uses_target_head": ("load_logit(w_draft, dtype, v * D + d)", "load_logit(w_target, dtype, v * D + d)",
                                      check_lmhead_integer_products),
    # n-gram pool: an n-gram already held is not inserted again
    "ngram_no_dedup": ("if (dup) continue;", "if (0) continue;", check_ngram_golden),
    # a full key drops its oldest n-gram, not its newest
    "ngram_evict_newest": ("if (oldest < 0 || l->e[i].stamp < l->e[oldest].stamp) oldest = i;",
                           "if (oldest < 0 || l->e[i].stamp > l->e[oldest].stamp) oldest = i;", check_ngram_golden),
    # only n-grams whose first token is the last generated token are candidates
    "ngram_no_first_token_filter": ("if (l->e[i].key == key && l->e[i].stamp < prev",
                                    "if (l->e[i].stamp < prev", check_ngram_properties),
    # candidates newest first
    "ngram_oldest_first": ("(best < 0 || l->e[i].stamp > l->e[best].stamp)",
                           "(best < 0 || l->e[i].stamp < l->e[best].stamp)", check_ngram_golden),
    # unused slots copy the newest candidate (or repeat the key)
    "ngram_pad_zeros": ("c > 0 ? out[t] : key;", "0;", check_ngram_golden),
    "multidraft_row_of_draft_0": ("load_row(target, dtype, (b * G + lead) * N + n, V, l);",
                                  "load_row(target, dtype, (b * G + 0) * N + n, V, l);", check_multidraft_marginal),
}


@pytest.fixture(scope="module")
def tmpdir_mod():
    with tempfile.TemporaryDirectory() as d:
        yield d


# The oracle function each mutation is planted in; the anchor must occur
# exactly once within that function's body.
FUNCTIONS = ("oracle_verify_sample", "oracle_row_stats", "oracle_verify_greedy", "oracle_verify_lookahead_sample",
             "oracle_verify_multidraft_sample", "oracle_verify_sample_lmhead", "oracle_inverse_cdf",
             "oracle_residual_draw", "oracle_ngram_pool_insert", "oracle_ngram_pool_lookup")


def function_span(src: str, fn: str):
    """[start, end) of the definition of ``fn`` in the oracle source."""
    start = src.index(f"\nint {fn}(")
    ends = [src.find(f"\nint {g}(", start + 1) for g in FUNCTIONS]
    ends = [e for e in ends if e > start]
    return start, min(ends) if ends else len(src)


def function_of(name: str) -> str:
    if name.startswith("lookahead_"):
        return "oracle_verify_lookahead_sample"
    if name.startswith("multidraft_"):
        return "oracle_verify_multidraft_sample"
    if name.startswith("lmhead_"):
        return "oracle_verify_sample_lmhead"
    if name.startswith(("argmax_", "greedy_")):
        return "oracle_verify_greedy"
    if name in ("ngram_no_dedup", "ngram_evict_newest"):
        return "oracle_ngram_pool_insert"
    if name.startswith("ngram_"):
        return "oracle_ngram_pool_lookup"
    return "oracle_verify_sample"


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pin_rejects_planted_mistake(name, tmpdir_mod):
    old, new, check = MUTATIONS[name]
    src = open(SRC).read()
    fn = function_of(name)
    if name in ("argmax_highest_index", "no_renormalise", "residual_sign", "zero_residual_from_q",
                "past_end_last_index", "past_end_first_positive"):  # helpers shared by the modes
        a, b = 0, len(src)
    else:
        a, b = function_span(src, fn)
    body = src[a:b]
    assert body.count(old) == 1, f"mutation anchor for {name} must occur exactly once in {fn}"
    path = os.path.join(tmpdir_mod, f"oracle_{name}.c")
    with open(path, "w") as f:
        f.write(src[:a] + body.replace(old, new) + src[b:])
    lib = oracle.load_library(oracle.compile_oracle(path, os.path.join(tmpdir_mod, f"lib_{name}.so")))
    with pytest.raises(AssertionError):
        check(lib)
