"""The CPU oracle of the multi-draft sampling verify against what the pages
and the mathematics fix (no GPU): each rejection step is the single-draft
rule of "Speculative Decoding —— LLM推理优化技术（一）" §2.1-2.2, so every
emitted token follows the target however many drafts are tried; one-hot
drafts give the Lookahead verify ("Lookahead Decoding 完全拆解", section
"采样模式的验证") and one draft the sampling-mode verify."""
import numpy as np
import pytest

import oracle
import specgen as sg

from pins import (check_multidraft_golden, check_multidraft_marginal, check_multidraft_one_hot_is_lookahead,
                  check_multidraft_single_draft_is_sampling, multidraft_case)


@pytest.fixture(scope="module")
def lib():
    return oracle._lib()


def test_one_hot_drafts_are_the_lookahead_verify(lib):
    check_multidraft_one_hot_is_lookahead(lib)


def test_one_draft_is_the_sampling_verify(lib):
    check_multidraft_single_draft_is_sampling(lib)


@pytest.mark.parametrize("T", [0.9, 1.4])
def test_marginal_law(lib, T):
    check_multidraft_marginal(lib, T)


def test_hand_cases(lib):
    check_multidraft_golden(lib)


def test_more_drafts_accept_more(lib):
    # every extra draft is one more chance at each position (the page's point
    # about adding draft sequences), with the output law unchanged
    lt, target, draft, toks, U = multidraft_case(100_000, 0.9, 34)
    _, acc3, _, _ = oracle.verify_multidraft_sample(target, draft, toks, U, 0.9, lib=lib)
    # draft 0's accept tests (u[n*G + 0]) and the draw uniform
    U1 = np.ascontiguousarray(np.concatenate([U[:, :-1].reshape(-1, 2, 3)[:, :, 0], U[:, -1:]], axis=1))
    _, acc1, _, _ = oracle.verify_multidraft_sample(target[:, :1], draft[:, :1], toks[:, :1], U1, 0.9, lib=lib)
    assert acc3.mean() > acc1.mean() + 0.05, (acc3.mean(), acc1.mean())


def test_input_errors_flag_the_sequence(lib):
    lt, target, draft, toks, U = multidraft_case(5, 1.0, 35)
    toks = toks.copy()
    toks[0, 1, 0] = 99            # token id out of range
    U[1, 2] = -0.5                # uniform outside [0, 1)
    draft[2, 2, 1, 3] = np.nan    # NaN in a draft row
    target[3, 1, 2, :] = -np.inf  # a target row of -inf only
    out, acc, best, _ = oracle.verify_multidraft_sample(target, draft, toks, U, 1.0, lib=lib)
    assert acc[:4].tolist() == [-1] * 4 and (out[:4] == -1).all() and (best[:4] == -1).all()
    assert acc[4] >= 0
    with pytest.raises(ValueError):
        oracle.verify_multidraft_sample(target, draft, toks, U, 0.0, lib=lib)


def test_workload_layout_and_shards(lib):
    cfg = sg.MULTIDRAFT_CONFIGS["md_sample_v32000_bf16"].with_(B=80, V=500)
    d = sg.multidraft_inputs(cfg)
    part = sg.multidraft_inputs(cfg, seq_offset=30, B=25)
    for k in d:
        np.testing.assert_array_equal(d[k][30:55], part[k])
    out, acc, best, _ = oracle.verify_multidraft_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                                        cfg.temperature, lib=lib)
    assert (acc >= 0).all()
    x = d["draft_tokens"]
    for b in range(cfg.B):
        j, g = acc[b], best[b]
        assert (out[b, :j] == x[b, g, :j]).all()
        assert not any((x[b, h, :j] == out[b, :j]).all() for h in range(g))
        assert 0 <= out[b, j] < cfg.V and (out[b, j + 1:] == -1).all()
        if j < cfg.N - 1:
            # after every still-matching draft is rejected, the residual is zero
            # at each of their tokens, so the drawn token is none of them
            held = {int(x[b, h, j]) for h in range(cfg.G) if (x[b, h, :j] == out[b, :j]).all()}
            assert int(out[b, j]) not in held
    assert len(set(acc.tolist())) >= 3
