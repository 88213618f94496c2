"""The CPU oracle of the Lookahead sampling-mode verify against what the page
and the mathematics fix (no GPU). Source: "Lookahead Decoding 完全拆解",
section "采样模式的验证": greedily produced candidates carry a one-hot draft
distribution, and the verify keeps the target's output distribution."""
import numpy as np
import pytest

import oracle
import specgen as sg

from pins import (check_lookahead_chisquare, check_lookahead_exact, check_lookahead_golden,
                  check_lookahead_single_candidate, lookahead_law, F)


@pytest.fixture(scope="module")
def lib():
    return oracle._lib()


def test_law_sums_to_one_and_reduces_to_one_candidate():
    # one candidate: the law is the autoregressive product along the candidate
    P = [[[F(1, 2), F(1, 2)], [F(1, 4), F(3, 4)]]]
    law = lookahead_law(P, [[1]])
    assert law == {(0, 0): F(1, 2), (1, 1, 0): F(1, 8), (1, 1, 1): F(3, 8)}


@pytest.mark.parametrize("shape", ["shared", "split"])
@pytest.mark.parametrize("dtype", [sg.F32, sg.BF16])
def test_exact_law_on_a_grid(lib, shape, dtype):
    check_lookahead_exact(lib, shape, dtype)


def test_law_by_chisquare(lib):
    check_lookahead_chisquare(lib)


def test_single_candidate_is_sampling_verify_with_one_hot_draft(lib):
    check_lookahead_single_candidate(lib)


def test_hand_cases(lib):
    check_lookahead_golden(lib)


def test_input_errors_flag_the_sequence(lib):
    cfg = sg.LOOKAHEAD_CONFIGS["la_sample_v32000_bf16"].with_(B=6, V=64)
    d = sg.lookahead_sample_inputs(cfg)
    L, C, U = d["logits"].copy(), d["cand"].copy(), d["uniforms"].copy()
    C[0, 3, 1] = cfg.V          # token id out of range
    U[1, 5] = 1.0               # uniform outside [0, 1)
    L[2, 6, 4, 7] = 0x7FC0      # NaN, in a row the walk may never reach
    L[3, 2, 1, :] = 0xFF80      # an all -inf row
    L[4, 0, 0, 9] = 0x7F80      # +inf
    out, acc, best, _ = oracle.verify_lookahead_sample(L, C, U, cfg.temperature, lib=lib)
    assert acc[:5].tolist() == [-1] * 5 and (out[:5] == -1).all() and (best[:5] == -1).all()
    assert acc[5] >= 0
    with pytest.raises(ValueError):
        oracle.verify_lookahead_sample(L, C, U, 0.0, lib=lib)


def test_output_layout(lib):
    cfg = sg.LOOKAHEAD_CONFIGS["la_sample_v32000_bf16"].with_(B=200, V=300, temperature=0.5)
    d = sg.lookahead_sample_inputs(cfg)
    out, acc, best, _ = oracle.verify_lookahead_sample(d["logits"], d["cand"], d["uniforms"], cfg.temperature,
                                                       lib=lib)
    assert (acc >= 0).all()
    for b in range(cfg.B):
        j, g = acc[b], best[b]
        assert 0 <= g < cfg.G and 0 <= j <= cfg.N - 1
        # the accepted prefix is the owner's, and no lower candidate matches it
        assert out[b, :j].tolist() == d["cand"][b, g, :j].tolist()
        assert all(d["cand"][b, h, :j].tolist() != out[b, :j].tolist() for h in range(g))
        assert 0 <= out[b, j] < cfg.V and (out[b, j + 1:] == -1).all()
        if j < cfg.N - 1:
            # the drawn token is none of the still-matching candidates' tokens
            held = {int(d["cand"][b, h, j]) for h in range(cfg.G) if d["cand"][b, h, :j].tolist() == out[b, :j].tolist()}
            assert int(out[b, j]) not in held
    assert len(set(acc.tolist())) >= 3, "the workload should reach several accept lengths"
