"""Helpers shared by the GPU tests: moving generated inputs to the device and
comparing the library against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg

NEAR_TIE = 1e-6  # |u - alpha|, CDF gap / Z, top-p cumulative gap


def dev():
    return torch.device("cuda", 0)


def to_dev(a: np.ndarray, device=None) -> torch.Tensor:
    device = device or dev()
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def run_sample(d: dict, temperature: float, top_p: float = 1.0, row_stats: bool = False):
    res = svpkg.verify_sample(to_dev(d["target"]), to_dev(d["draft"]), to_dev(d["draft_tokens"]),
                              to_dev(d["uniforms"]), temperature, top_p, row_stats=row_stats)
    torch.cuda.synchronize()
    return tuple(r.cpu().numpy() for r in res)


def compare_sample(d: dict, temperature: float, top_p: float = 1.0, gpu=None, max_mismatch: int | None = 0):
    """Tokens and accept lengths must equal the oracle's, except in sequences
    whose smallest decision margin is below NEAR_TIE (a near-tie: |u - alpha|,
    the draw's CDF gap over Z, or a top-p cumulative gap). Mismatches are only
    allowed at near-ties, and at most ``max_mismatch`` of them (None: no cap,
    for rate measurements). Returns a summary with the counts."""
    if gpu is None:
        gpu = run_sample(d, temperature, top_p)
    gt, ga = gpu[0], gpu[1]
    rt, ra, margin = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], temperature,
                                          top_p)
    diff = (ga != ra) | (gt != rt).any(1)
    near = margin < NEAR_TIE
    bad = diff & ~near
    i = int(np.argmax(bad))
    assert not bad.any(), (
        f"{int(bad.sum())} sequences differ from the oracle away from a near-tie; first: b={i} "
        f"gpu {gt[i]} / {ga[i]} oracle {rt[i]} / {ra[i]} margin {margin[i]}")
    K = d["draft_tokens"].shape[1]
    decisions = int(np.where(ra >= 0, np.minimum(ra + 1, K) + 1, 0).sum())
    if max_mismatch is not None:
        assert diff.sum() <= max_mismatch, (int(diff.sum()), decisions)
    return {"sequences": len(ra), "mismatch": int(diff.sum()), "near_ties": int(near.sum()),
            "decisions": decisions, "accept_mean": float(ra[ra >= 0].mean()) if (ra >= 0).any() else 0.0}


def compare_row_stats(d: dict, stats: np.ndarray, temperature: float, top_p: float, rows=None):
    """GPU row stats {m, lse, P_S, tau} against the oracle's fp64 values:
    m, lse and P_S within 1e-5 relative; tau exact unless the nucleus cut is a
    near-tie (then both cuts must hold top_p within 1e-5)."""
    B, K1, V = d["target"].shape
    K = K1 - 1
    allrows = np.concatenate([d["target"], d["draft"]], axis=1)  # [B, 2K+1, V]
    flat = allrows.reshape(-1, V)
    st = stats.reshape(-1, 4)
    idx = np.arange(flat.shape[0]) if rows is None else np.asarray(rows)
    ref = oracle.row_stats(flat[idx], temperature, top_p)
    g = st[idx].astype(np.float64)
    same_cut = g[:, 3] == ref[:, 3]
    for col, name in ((0, "m"), (1, "lse"), (2, "P_S")):
        err = np.abs(g[:, col] - ref[:, col]) / np.maximum(1.0, np.abs(ref[:, col]))
        if col == 2:
            err = np.where(same_cut, err, 0.0)
        assert err.max() <= 1e-5, (name, float(err.max()), int(idx[np.argmax(err)]))
    if top_p < 1.0:
        vals = sg.to_float(flat[idx], sg.BF16 if d["target"].dtype == np.uint16 else sg.F32)
        for k in np.nonzero(~same_cut)[0]:
            z = vals[k] / np.float64(np.float32(temperature))
            p = np.exp(z - z.max())
            p /= p.sum()
            for tau in (g[k, 3], ref[k, 3]):
                assert abs(p[vals[k] >= tau].sum() - top_p) < 1e-5 or p[vals[k] > tau].sum() < top_p <= p[
                    vals[k] >= tau].sum(), (int(idx[k]), g[k, 3], ref[k, 3])
    else:
        assert np.all(g[:, 3] == -np.inf)


def run_greedy(d: dict):
    res = svpkg.verify_greedy(to_dev(d["logits"]), to_dev(d["cand"]), best=True)
    torch.cuda.synchronize()
    return tuple(r.cpu().numpy() for r in res)


def compare_greedy(d: dict):
    gt, ga, gb = run_greedy(d)
    rt, ra, rb = oracle.verify_greedy(d["logits"], d["cand"])
    np.testing.assert_array_equal(ga, ra)
    np.testing.assert_array_equal(gt, rt)
    np.testing.assert_array_equal(gb, rb)
    return {"sequences": len(ra), "accept_mean": float(ra[ra >= 0].mean()) if (ra >= 0).any() else 0.0}


def run_lookahead(d: dict, temperature: float, row_lse: bool = False):
    res = svpkg.verify_lookahead_sample(to_dev(d["logits"]), to_dev(d["cand"]), to_dev(d["uniforms"]), temperature,
                                        best=True, row_lse=row_lse)
    torch.cuda.synchronize()
    return tuple(r.cpu().numpy() for r in res)


def compare_lookahead(d: dict, temperature: float, gpu=None, max_mismatch: int | None = 0):
    """Lookahead sampling verify: tokens, accept lengths and owners equal the
    oracle's except in sequences whose smallest decision margin (|u - alpha|
    of a test, CDF gap / Z of the draw) is below NEAR_TIE; at most
    ``max_mismatch`` such sequences differ. Returns counts."""
    if gpu is None:
        gpu = run_lookahead(d, temperature)
    gt, ga, gb = gpu[0], gpu[1], gpu[2]
    rt, ra, rb, margin = oracle.verify_lookahead_sample(d["logits"], d["cand"], d["uniforms"], temperature)
    diff = (ga != ra) | (gb != rb) | (gt != rt).any(1)
    near = margin < NEAR_TIE
    bad = diff & ~near
    i = int(np.argmax(bad))
    assert not bad.any(), (
        f"{int(bad.sum())} sequences differ from the oracle away from a near-tie; first: b={i} "
        f"gpu {gt[i]} / {ga[i]} / {gb[i]} oracle {rt[i]} / {ra[i]} / {rb[i]} margin {margin[i]}")
    if max_mismatch is not None:
        assert diff.sum() <= max_mismatch, int(diff.sum())
    return {"sequences": len(ra), "mismatch": int(diff.sum()), "near_ties": int(near.sum()),
            "accept_hist": np.bincount(ra[ra >= 0], minlength=d["cand"].shape[2] + 1).tolist()}


def run_multidraft(d: dict, temperature: float, row_lse: bool = False):
    res = svpkg.verify_multidraft_sample(to_dev(d["target"]), to_dev(d["draft"]), to_dev(d["draft_tokens"]),
                                         to_dev(d["uniforms"]), temperature, best=True, row_lse=row_lse)
    torch.cuda.synchronize()
    return tuple(r.cpu().numpy() for r in res)


def compare_multidraft(d: dict, temperature: float, gpu=None, max_mismatch: int | None = 0):
    """Multi-draft sampling verify against the oracle, with the same near-tie
    rule as compare_lookahead."""
    if gpu is None:
        gpu = run_multidraft(d, temperature)
    gt, ga, gb = gpu[0], gpu[1], gpu[2]
    rt, ra, rb, margin = oracle.verify_multidraft_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                                         temperature)
    diff = (ga != ra) | (gb != rb) | (gt != rt).any(1)
    near = margin < NEAR_TIE
    bad = diff & ~near
    i = int(np.argmax(bad))
    assert not bad.any(), (
        f"{int(bad.sum())} sequences differ from the oracle away from a near-tie; first: b={i} "
        f"gpu {gt[i]} / {ga[i]} / {gb[i]} oracle {rt[i]} / {ra[i]} / {rb[i]} margin {margin[i]}")
    if max_mismatch is not None:
        assert diff.sum() <= max_mismatch, int(diff.sum())
    return {"sequences": len(ra), "mismatch": int(diff.sum()), "near_ties": int(near.sum())}
