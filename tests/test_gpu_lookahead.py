"""GPU parity of the Lookahead sampling-mode verify ("Lookahead Decoding 完全拆解",
section "采样模式的验证") against the CPU oracle, through the C ABI: tokens,
accept lengths and owners identical except at near-ties (|u - alpha| or CDF
gap / Z below 1e-6); row log-normalisers within 1e-5."""
import numpy as np
import pytest
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg
from gpu_util import compare_lookahead, run_lookahead, to_dev

pytestmark = pytest.mark.gpu

LA = sg.LOOKAHEAD_CONFIGS["la_sample_v32000_bf16"]


@pytest.fixture(scope="module", autouse=True)
def built():
    svpkg.build()
    torch.cuda.set_device(0)
    yield
    assert svpkg.get_status() == 0


CASES = {
    # small and ragged: rows not 16-byte aligned, heads and tails on every row
    "bf16_v1001_g7_n5_t05": LA.with_(B=50, V=1001, temperature=0.5, seed=1),
    "f32_v3001_g3_n4_t07": LA.with_(B=40, V=3001, G=3, N=4, dtype=sg.F32, temperature=0.7, seed=2),
    # many candidates, most sharing their first token
    "bf16_v517_g12_n3": LA.with_(B=60, V=517, G=12, N=3, match_prob=0.8, temperature=0.4, seed=3),
    # one candidate: every position is a one-hot sampling verify
    "bf16_v2000_g1_n6": LA.with_(B=60, V=2000, G=1, N=6, match_prob=0.9, temperature=0.3, seed=4),
    # the per-sequence limits: G = 32 (one warp), and G*N = 1024
    "bf16_v700_g32_n5": LA.with_(B=10, V=700, G=32, N=5, match_prob=0.9, temperature=0.3, seed=5),
    "f32_v300_g4_n256": LA.with_(B=3, V=300, G=4, N=256, dtype=sg.F32, match_prob=0.97, temperature=0.2, seed=6),
    # N = 2: one position and the bonus
    "bf16_v5000_g5_n2": LA.with_(B=64, V=5000, G=5, N=2, temperature=0.6, seed=7),
    # a row longer than one thread's chunk per 512 threads many times over
    "bf16_v151936_g4_n3": LA.with_(B=6, V=151936, G=4, N=3, temperature=0.5, seed=8),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_lookahead_parity(name):
    cfg = CASES[name]
    d = sg.lookahead_sample_inputs(cfg)
    gt, ga, gb, gl = run_lookahead(d, cfg.temperature, row_lse=True)
    compare_lookahead(d, cfg.temperature, gpu=(gt, ga, gb), max_mismatch=1)
    ref = oracle.row_stats(d["logits"].reshape(-1, cfg.V), cfg.temperature)[:, 1]
    err = np.abs(gl.reshape(-1).astype(np.float64) - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() <= 1e-5, float(err.max())


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_full_size_lookahead(T):
    cfg = LA.with_(temperature=T)
    d = sg.lookahead_sample_inputs(cfg)
    compare_lookahead(d, T, max_mismatch=1)


def test_lookahead_bad_inputs_flag_only_their_sequence():
    cfg = LA.with_(B=8, V=900, temperature=0.6)
    d = sg.lookahead_sample_inputs(cfg)
    d["cand"][0, 3, 1] = cfg.V
    d["cand"][1, 0, 0] = -2
    d["uniforms"][2, 5] = 1.0
    d["logits"][3, 6, 4, 7] = 0x7FC0    # NaN in a row the walk may never reach
    d["logits"][4, 2, 1, :] = 0xFF80    # a row of -inf only
    d["logits"][5, 0, 0, 9] = 0x7F80    # +inf
    gt, ga, gb = run_lookahead(d, cfg.temperature)
    assert svpkg.get_status() == -4
    assert svpkg.get_status() == 0
    assert (ga[:6] == -1).all() and (gt[:6] == -1).all() and (gb[:6] == -1).all()
    compare_lookahead(d, cfg.temperature, gpu=(gt, ga, gb))


def test_lookahead_hand_cases():
    import os
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    from pins import load_lookahead_golden
    for logits, cand, u, T, toks, acc, best in load_lookahead_golden():
        gt, ga, gb = run_lookahead({"logits": logits, "cand": cand, "uniforms": u}, T)
        assert gt[0].tolist() == toks and ga[0] == acc and gb[0] == best, (gt, ga, gb, toks, acc, best)


def test_lookahead_host_buffers_and_repeat():
    cfg = LA.with_(B=16, V=6000, temperature=0.5, seed=9)
    d = sg.lookahead_sample_inputs(cfg)
    a = run_lookahead(d, cfg.temperature)
    b = run_lookahead(d, cfg.temperature)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)

    def host(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
        return torch.from_numpy(x).pin_memory()

    ht, ha, hb = svpkg.verify_lookahead_sample(host(d["logits"]), host(d["cand"]), host(d["uniforms"]),
                                               cfg.temperature, best=True)
    assert ht.device.type == "cpu"
    np.testing.assert_array_equal(ht.numpy(), a[0])
    np.testing.assert_array_equal(ha.numpy(), a[1])
    np.testing.assert_array_equal(hb.numpy(), a[2])


def test_lookahead_between_other_calls_on_one_stream():
    # the three entry points share the stream's scratch area
    s = sg.sample_inputs(sg.CONFIGS["cfg2_v32000_bf16"].with_(B=4, V=3000))
    g = sg.greedy_inputs(sg.CONFIGS["cfg4_greedy_v32000_bf16"].with_(B=4, V=3000))
    la = sg.lookahead_sample_inputs(LA.with_(B=20, V=3000, temperature=0.5))
    first = run_lookahead(la, 0.5)
    svpkg.verify_sample(to_dev(s["target"]), to_dev(s["draft"]), to_dev(s["draft_tokens"]), to_dev(s["uniforms"]),
                        1.0)
    again = run_lookahead(la, 0.5)
    svpkg.verify_greedy(to_dev(g["logits"]), to_dev(g["cand"]))
    third = run_lookahead(la, 0.5)
    for x, y, z in zip(first, again, third):
        np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(x, z)
    compare_lookahead(la, 0.5, gpu=first)
