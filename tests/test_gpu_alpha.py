"""The accept probabilities, element by element, through the accept decisions.

alpha_i = min(1, p'_i(x_i) / q'_i(x_i)) ("Speculative Decoding —— LLM推理优化技术（一）"
§2.1; kwkr.cn "投机解码" §3.1) uses the logits of the draft token in the target
and draft rows (gathered by the kernels), the rows' normalisers and, with
top-p, their nucleus masses and cuts. Here every uniform is placed 1e-4
(relative) inside or outside the oracle's alpha: u_i = alpha_i (1 - 1e-4) before
a chosen position j, u_j = alpha_j (1 + 1e-4) at it. A gathered logit, a
normaliser or a cut that is off by more than about 1e-4 flips a decision, so
the accept lengths must equal the oracle's exactly, sequence by sequence.
alpha_i itself comes from the oracle's row statistics:
p'(x) = exp(l_x / T - lse) / P_S on the nucleus {l >= tau}, else 0."""
import numpy as np
import pytest
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg
from gpu_util import run_sample

pytestmark = pytest.mark.gpu

C = sg.CONFIGS


@pytest.fixture(scope="module", autouse=True)
def built():
    svpkg.build()
    torch.cuda.set_device(0)
    yield
    assert svpkg.get_status() == 0


def _alpha(d, T, top_p, dtype):
    """Oracle alpha[B, K] from the oracle's row statistics {m, lse, P_S, tau}."""
    tgt, dft, x = d["target"], d["draft"], d["draft_tokens"]
    B, K = x.shape
    sp = oracle.row_stats(tgt[:, :K], T, top_p)  # [B, K, 4]
    sq = oracle.row_stats(dft, T, top_p)
    bi, ki = np.meshgrid(np.arange(B), np.arange(K), indexing="ij")
    # the stored logits (bf16 rows hold raw 16-bit patterns)
    lp = sg.to_float(tgt[bi, ki, x], dtype).astype(np.float64)
    lq = sg.to_float(dft[bi, ki, x], dtype).astype(np.float64)

    def prob(l, s):
        p = np.exp(l / T - s[..., 1]) / s[..., 2]
        return np.where(l >= s[..., 3], p, 0.0)

    p, q = prob(lp, sp), prob(lq, sq)
    with np.errstate(divide="ignore", invalid="ignore"):
        a = np.where(p == 0, 0.0, np.where(q == 0, 1.0, np.minimum(1.0, p / q)))
    return a


CASES = {
    "cfg2_b64": (C["cfg2_v32000_bf16"].with_(B=64), 2),
    "cfg2_b64_streaming": (C["cfg2_v32000_bf16"].with_(B=64), 1),
    "cfg1_b300_f32": (C["cfg1_v1000_f32"].with_(B=300), 0),
    "cfg3_b16": (C["cfg3_v128256_bf16"].with_(B=16), 0),
    "cfg5_b16_topp": (C["cfg5_topp_v151936_bf16"].with_(B=16), 0),
    "cfg5_b16_topp_streaming": (C["cfg5_topp_v151936_bf16"].with_(B=16), 1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_accept_decisions_pin_alpha(name):
    cfg, path = CASES[name]
    d = sg.sample_inputs(cfg)
    B, K = d["draft_tokens"].shape
    a = _alpha(d, cfg.temperature, cfg.top_p, cfg.dtype)
    assert np.isfinite(a).all() and (a >= 0).all() and (a <= 1).all()
    rng = np.random.default_rng(11)
    j = rng.integers(0, K + 1, size=B)  # the position to reject at (K: accept all)
    u = d["uniforms"].astype(np.float64).copy()
    pos = np.arange(K)[None, :]
    below = a * (1 - 1e-4)
    above = np.minimum(a * (1 + 1e-4), 1 - 2.0 ** -24)
    u[:, :K] = np.where(pos < j[:, None], below, np.where(pos == j[:, None], above, u[:, :K]))
    d["uniforms"] = u.astype(np.float32)
    svpkg.set_sample_path(path)
    try:
        gt, ga = run_sample(d, cfg.temperature, cfg.top_p)[:2]
    finally:
        svpkg.set_sample_path(0)
    rt, ra, _ = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], cfg.temperature,
                                     cfg.top_p)
    bad = np.nonzero(ga != ra)[0]
    assert bad.size == 0, (f"{bad.size} accept lengths differ; first b={bad[0]}: gpu {ga[bad[0]]} oracle "
                           f"{ra[bad[0]]} alpha {a[bad[0]]}")
    # and the decisions were the intended ones: every sequence stops at j or
    # earlier (an alpha of 0), or later only where alpha_j is 1
    late = ra > j
    assert (a[late, j[late]] == 1.0).all()
