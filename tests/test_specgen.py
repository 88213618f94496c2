"""The seeded input generator: Philox known answers, shard invariance, and the
draft sampler's marginal distribution."""
import os

import numpy as np
import pytest
from scipy import stats

import specgen as sg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        assert sg.philox4x32_10(v[0:4], v[4:6]) == tuple(v[6:10])


def test_shards_equal_whole_batch():
    cfg = sg.CONFIGS["cfg2_v32000_bf16"].with_(B=6, V=777)
    whole = sg.sample_inputs(cfg)
    a = sg.sample_inputs(cfg, seq_offset=0, B=2)
    b = sg.sample_inputs(cfg, seq_offset=2, B=4)
    for k in whole:
        np.testing.assert_array_equal(whole[k], np.concatenate([a[k], b[k]]))
    g = sg.CONFIGS["cfg4_greedy_v32000_bf16"].with_(B=5, V=300)
    gw = sg.greedy_inputs(g)
    g1, g2 = sg.greedy_inputs(g, 0, 3), sg.greedy_inputs(g, 3, 2)
    for k in gw:
        np.testing.assert_array_equal(gw[k], np.concatenate([g1[k], g2[k]]))


def test_thread_count_does_not_change_bytes():
    cfg = sg.CONFIGS["cfg5_topp_v151936_bf16"].with_(B=3, V=2000)
    a = sg.sample_inputs(cfg, nthreads=1)
    b = sg.sample_inputs(cfg, nthreads=3)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_logit_statistics_follow_the_recipe():
    cfg = sg.CONFIGS["cfg3_v128256_bf16"].with_(B=2, V=20000)
    d = sg.sample_inputs(cfg)
    t = sg.to_float(d["target"], cfg.dtype)
    dr = sg.to_float(d["draft"], cfg.dtype)
    # n_peaks entries per row lifted by peak_height: the row maximum sits well above the noise
    assert abs(np.median(t) - 0.0) < 0.05 and abs(np.std(t) - cfg.target_sigma) < 0.05
    diff = dr - t[:, : cfg.K]
    assert abs(np.std(diff) - cfg.draft_sigma) < 0.05
    assert d["uniforms"].min() >= 0 and d["uniforms"].max() < 1
    assert d["draft_tokens"].min() >= 0 and d["draft_tokens"].max() < cfg.V


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.6, 1.0), (1.0, 0.75)])
def test_draft_sampler_marginal(T, top_p):
    """Draft tokens are draws from softmax(l/T) restricted to the nucleus."""
    V, n = 7, 200_000
    l = np.array([1.2, -0.3, 0.8, 2.0, 0.0, -1.5, 0.8], dtype=np.float32)
    draft = np.broadcast_to(l, (n, 1, V)).copy()
    toks = sg.draft_tokens(draft, sg.F32, T, top_p, seed=3)
    z = l.astype(np.float64) / T
    q = np.exp(z - z.max())
    q /= q.sum()
    if top_p < 1:
        # brute force over thresholds: the largest tau whose upper set holds >= top_p
        taus = sorted(set(l.tolist()), reverse=True)
        tau = next(t for t in taus if q[l >= t].sum() >= top_p)
        q = np.where(l >= tau, q, 0.0)
        q /= q.sum()
    counts = np.bincount(toks.ravel(), minlength=V)
    keep = q > 0
    assert counts[~keep].sum() == 0
    _, pval = stats.chisquare(counts[keep], q[keep] * n)
    assert pval > 1e-3


def test_greedy_candidates_match_argmax_then_random():
    cfg = sg.CONFIGS["cfg4_greedy_v32000_bf16"].with_(B=400, V=64)
    d = sg.greedy_inputs(cfg)
    a = sg.to_float(d["logits"], cfg.dtype).argmax(-1)  # numpy argmax: first maximum
    hit = d["cand"] == a[:, :, : cfg.N - 1]
    first = hit[..., 0].mean()
    assert abs(first - (0.5 + 0.5 / cfg.V)) < 0.02
