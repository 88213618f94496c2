"""The verify on hidden states (sv_verify_sample_lmhead): the tcgen05 GEMM's
logits against numpy's h @ W.T, and the tokens against the oracle's verify on
fp64 logits (oracle_verify_sample_lmhead). Hidden states and heads hold small
integers, so every product and every partial sum is exact in fp32 and the
two sides see the same logits."""
import numpy as np
import pytest
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg
from gpu_util import NEAR_TIE, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    svpkg.build()
    torch.cuda.set_device(0)
    yield
    assert svpkg.get_status() == 0


def make(B, K, D, V, T, seed):
    rng = np.random.default_rng(seed)
    ht = rng.integers(-3, 4, size=(B, K + 1, D)).astype(np.float32)
    hd = rng.integers(-3, 4, size=(B, K, D)).astype(np.float32)
    wt = rng.integers(-2, 3, size=(V, D)).astype(np.float32)
    wd = rng.integers(-2, 3, size=(V, D)).astype(np.float32)
    lt = ht.astype(np.float64) @ wt.T.astype(np.float64)
    ld = hd.astype(np.float64) @ wd.T.astype(np.float64)
    toks = sg.draft_tokens(ld.astype(np.float32), sg.F32, T, 1.0, seed=seed)
    U = sg.uniforms(B, K, seed=seed)
    bf = lambda a: sg.from_float(a, sg.BF16)  # integers in [-3, 3] are exact in bf16
    return bf(ht), bf(hd), bf(wt), bf(wd), lt, ld, toks, U


# (shapes: one, two and three 128-row tiles of positions per pass; more rows
# than one pass takes (500 target rows: a pass of 384, then 116); ragged V)
@pytest.mark.parametrize("B,K,D,V,T", [(4, 3, 128, 1000, 3.0), (40, 5, 256, 4099, 6.0), (1, 1, 64, 130, 2.0),
                                       (64, 5, 512, 32000, 16.0), (100, 4, 128, 700, 4.0)])
def test_lmhead_logits_and_verify(B, K, D, V, T):
    ht, hd, wt, wd, lt, ld, toks, U = make(B, K, D, V, T, seed=B + D)
    out_t, out_a, lg = svpkg.verify_sample_lmhead(to_dev(ht), to_dev(hd), to_dev(wt), to_dev(wd), to_dev(toks),
                                                  to_dev(U), T, logits=True)
    torch.cuda.synchronize()
    lg = lg.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(lg[:B * (K + 1)], lt.reshape(-1, V))
    np.testing.assert_array_equal(lg[B * (K + 1):], ld.reshape(-1, V))
    rt, ra, margin = oracle.verify_sample_lmhead(ht, hd, wt, wd, toks, U, T)
    gt, ga = out_t.cpu().numpy(), out_a.cpu().numpy()
    diff = (ga != ra) | (gt != rt).any(1)
    assert not (diff & (margin >= NEAR_TIE)).any(), np.nonzero(diff)[0][:10]
    assert diff.sum() <= 1
    assert (ra >= 0).all()


def test_lmhead_argument_errors():
    lib = svpkg.lib()
    x = torch.zeros(1024, dtype=torch.int32, device="cuda")
    p = svpkg._ptr(x)
    # D not a multiple of 64
    assert lib.sv_verify_sample_lmhead(p, p, p, p, p, p, 2, 1, 100, 50, 1.0, 1.0, p, p, None, None) == -1
    # T = 0 has no meaning here
    assert lib.sv_verify_sample_lmhead(p, p, p, p, p, p, 2, 1, 64, 50, 0.0, 1.0, p, p, None, None) == -1
    assert lib.sv_verify_sample_lmhead(None, p, p, p, p, p, 2, 1, 64, 50, 1.0, 1.0, p, p, None, None) == -1
