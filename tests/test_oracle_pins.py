"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import math

import numpy as np
import pytest

import oracle
import specgen as sg

from pins import (LD, LT, check_acceptance_is_one_minus_tv, check_brute_force, check_draw_edge_rules,
                  check_greedy_golden,
                  check_greedy_multi_draft, check_output_is_target_distribution, check_tokens_per_round,
                  check_topp_golden, multi_draft_expected_tokens, nucleus_bruteforce, replicate, softmax)


@pytest.fixture(scope="module")
def lib():
    return oracle._lib()


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.7, 1.0), (1.0, 0.8), (1.3, 0.6)])
def test_output_follows_target(lib, T, top_p):
    check_output_is_target_distribution(lib, T, top_p)


def test_acceptance_rate(lib):
    check_acceptance_is_one_minus_tv(lib)


@pytest.mark.parametrize("K", [1, 4, 8])
def test_tokens_per_round(lib, K):
    check_tokens_per_round(lib, K)


@pytest.mark.parametrize("K", [1, 2])
def test_brute_force_joint_mass(lib, K):
    check_brute_force(lib, K=K)


def test_draw_edge_rules(lib):
    check_draw_edge_rules(lib)


def test_topp_golden(lib):
    check_topp_golden(lib)


def test_topp_bruteforce_random_rows(lib):
    rng = np.random.default_rng(7)
    for _ in range(300):
        V = int(rng.integers(2, 12))
        l = (rng.integers(-6, 7, size=V) / 4.0).astype(np.float32)  # many ties
        # the oracle takes T and top_p as fp32, so the brute force uses the same values
        T = float(np.float32(rng.choice([0.5, 1.0, 1.7])))
        top_p = float(np.float32(rng.choice([0.1, 0.5, 0.73, 0.9, 0.999])))
        st = oracle.row_stats(l[None], T, top_p, lib=lib)[0]
        p = softmax(l, T)
        tau = nucleus_bruteforce(l, p, top_p)
        assert st[3] == tau
        assert abs(st[2] - p[l >= tau].sum()) < 1e-12


def test_normalisers_exact(lib):
    rng = np.random.default_rng(8)
    for dt in (sg.F32, sg.BF16):
        x = rng.normal(0, 3, size=(5, 3001))
        x[0, :7] = -np.inf
        rows = sg.from_float(x, dt)
        for T in (float(np.float32(t)) for t in (0.3, 1.0, 2.5)):
            st = oracle.row_stats(rows, T, 1.0, lib=lib)
            vals = sg.to_float(rows, dt)
            for r in range(rows.shape[0]):
                z = vals[r] / T
                m = z.max()
                lse = m + math.log(math.fsum(np.exp(z - m).tolist()))
                assert st[r, 0] == m
                assert abs(st[r, 1] - lse) <= 1e-12 * max(1.0, abs(lse))
                assert st[r, 2] == 1.0 and st[r, 3] == -np.inf


def test_greedy_golden(lib):
    check_greedy_golden(lib)


def test_multi_draft_formula_matches_the_page():
    # eq. (5) with g = 4, b = 7, a = 0.5 (the greedy workload's shape)
    assert abs(multi_draft_expected_tokens(4, 7, 0.5) - 3.8295) < 1e-4
    # b = 1 reduces to the geometric series (1 - a^(g+1)) / (1 - a)
    assert abs(multi_draft_expected_tokens(4, 1, 0.6) - (1 - 0.6 ** 5) / 0.4) < 1e-12


def test_greedy_multi_draft(lib):
    check_greedy_multi_draft(lib)


def test_identical_distributions_always_accept(lib):
    n, K = 5000, 3
    rows = np.tile(LT[0], (K + 1, 1))
    target, draft = replicate(rows, rows[:K], n)
    toks = sg.draft_tokens(draft, sg.F32, 0.9, 1.0, seed=1)
    u = sg.uniforms(n, K, seed=1)
    _, acc, _ = oracle.verify_sample(target, draft, toks, u, 0.9, 1.0, lib=lib)
    assert (acc == K).all()


def test_disjoint_supports_always_reject(lib):
    n, V = 200_000, 6
    lt = np.array([[0.0, 1.0, 2.0, -np.inf, -np.inf, -np.inf]] * 2, np.float32)
    ld = np.array([[-np.inf, -np.inf, -np.inf, 0.5, 0.0, 1.0]], np.float32)
    target, draft = replicate(lt, ld, n)
    toks = sg.draft_tokens(draft, sg.F32, 1.0, 1.0, seed=2)
    u = sg.uniforms(n, 1, seed=2)
    out, acc, _ = oracle.verify_sample(target, draft, toks, u, 1.0, 1.0, lib=lib)
    assert (acc == 0).all()
    # the residual max(0, p - q) is p itself
    p = softmax(lt[0])
    c = np.bincount(out[:, 0], minlength=V)
    from scipy import stats
    _, pval = stats.chisquare(c[:3], p[:3] * n)
    assert pval > 1e-3 and c[3:].sum() == 0


def test_low_temperature_equals_greedy_limit(lib):
    # fp32 logits, so that no row has two equal maxima (with a tie the T -> 0
    # limit splits the mass, while T = 0 takes the lowest index)
    cfg = sg.CONFIGS["cfg2_v32000_bf16"].with_(B=50, V=500, temperature=0.0, dtype=sg.F32)
    d = sg.sample_inputs(cfg)
    out0, acc0, _ = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 0.0, lib=lib)
    out1, acc1, m = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 1e-3, lib=lib)
    assert (acc0 >= 0).all()
    np.testing.assert_array_equal(acc0, acc1)
    np.testing.assert_array_equal(out0, out1)


def test_input_errors_flag_the_sequence(lib):
    cfg = sg.CONFIGS["cfg2_v32000_bf16"].with_(B=6, V=64)
    d = sg.sample_inputs(cfg)
    t, dr, x, u = d["target"].copy(), d["draft"].copy(), d["draft_tokens"].copy(), d["uniforms"].copy()
    x[0, 2] = cfg.V             # token id out of range
    x[1, 0] = -1
    u[2, 1] = 1.0               # uniform outside [0, 1)
    t[3, 4, 5] = 0x7FC0         # NaN (bf16 pattern)
    dr[4, 0, :] = 0xFF80        # all -inf draft row
    out, acc, _ = oracle.verify_sample(t, dr, x, u, 1.0, lib=lib)
    assert acc[:5].tolist() == [-1] * 5 and (out[:5] == -1).all()
    assert acc[5] >= 0
    with pytest.raises(ValueError):
        oracle.verify_sample(t, dr, x, u, -1.0, lib=lib)
    with pytest.raises(ValueError):
        oracle.verify_sample(t, dr, x, u, 1.0, 0.0, lib=lib)


def test_output_layout(lib):
    cfg = sg.CONFIGS["cfg3_v128256_bf16"].with_(B=40, V=300)
    d = sg.sample_inputs(cfg)
    out, acc, _ = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], cfg.temperature,
                                       lib=lib)
    for b in range(cfg.B):
        j = acc[b]
        assert 0 <= j <= cfg.K
        assert out[b, :j].tolist() == d["draft_tokens"][b, :j].tolist()
        assert 0 <= out[b, j] < cfg.V
        assert (out[b, j + 1:] == -1).all()
