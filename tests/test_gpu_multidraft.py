"""GPU parity of the multi-draft sampling verify against the CPU oracle,
through the C ABI: tokens, accept lengths and owners identical except at
near-ties (|u - alpha| or CDF gap / Z below 1e-6); row log-normalisers within
1e-5."""
import numpy as np
import pytest
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg
from gpu_util import compare_multidraft, run_multidraft

pytestmark = pytest.mark.gpu

MD = sg.MULTIDRAFT_CONFIGS["md_sample_v32000_bf16"]


@pytest.fixture(scope="module", autouse=True)
def built():
    svpkg.build()
    torch.cuda.set_device(0)
    yield
    assert svpkg.get_status() == 0


CASES = {
    "bf16_v700_g7_n5": MD.with_(B=40, V=700, seed=1),
    "f32_v1501_g3_n4_t07": MD.with_(B=40, V=1501, G=3, N=4, dtype=sg.F32, temperature=0.7, seed=2),
    "bf16_v300_g12_n3_t05": MD.with_(B=30, V=300, G=12, N=3, temperature=0.5, seed=3),
    "bf16_v2000_g1_n6": MD.with_(B=30, V=2000, G=1, N=6, temperature=0.8, seed=4),
    "bf16_v500_g32_n3": MD.with_(B=6, V=500, G=32, N=3, seed=5),
    "bf16_v151936_g3_n3": MD.with_(B=4, V=151936, G=3, N=3, temperature=0.7, seed=6),
    # the walk with the position's distribution in shared memory: at its
    # largest row, and a row that is not a whole number of 16-byte vectors
    "bf16_v51200_g4_n4": MD.with_(B=8, V=51200, G=4, N=4, seed=7),
    "bf16_v32007_g7_n5": MD.with_(B=8, V=32007, seed=8),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_multidraft_parity(name):
    cfg = CASES[name]
    d = sg.multidraft_inputs(cfg)
    gt, ga, gb, gl = run_multidraft(d, cfg.temperature, row_lse=True)
    compare_multidraft(d, cfg.temperature, gpu=(gt, ga, gb), max_mismatch=1)
    rows = np.concatenate([d["target"].reshape(-1, cfg.V), d["draft"].reshape(-1, cfg.V)])
    ref = oracle.row_stats(rows, cfg.temperature)[:, 1]
    err = np.abs(gl.astype(np.float64) - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() <= 1e-5, float(err.max())


def test_full_size_multidraft():
    d = sg.multidraft_inputs(MD)
    compare_multidraft(d, MD.temperature, max_mismatch=1)


def test_one_hot_drafts_match_the_lookahead_path():
    cfg = sg.LOOKAHEAD_CONFIGS["la_sample_v32000_bf16"].with_(B=24, V=900, dtype=sg.F32, temperature=0.6)
    la = sg.lookahead_sample_inputs(cfg)
    draft = np.full(la["cand"].shape + (cfg.V,), -np.inf, np.float32)
    np.put_along_axis(draft, la["cand"][..., None], 0.0, axis=-1)
    dev = torch.device("cuda", 0)
    a = svpkg.verify_multidraft_sample(torch.from_numpy(la["logits"]).to(dev), torch.from_numpy(draft).to(dev),
                                       torch.from_numpy(la["cand"]).to(dev), torch.from_numpy(la["uniforms"]).to(dev),
                                       cfg.temperature, best=True)
    b = svpkg.verify_lookahead_sample(torch.from_numpy(la["logits"]).to(dev), torch.from_numpy(la["cand"]).to(dev),
                                      torch.from_numpy(la["uniforms"]).to(dev), cfg.temperature, best=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy())


def test_multidraft_bad_inputs_flag_only_their_sequence():
    cfg = MD.with_(B=6, V=800, temperature=0.9)
    d = sg.multidraft_inputs(cfg)
    d["draft_tokens"][0, 2, 1] = cfg.V
    d["uniforms"][1, 3] = 1.0
    d["draft"][2, 4, 2, 5] = 0x7FC0    # NaN in a draft row
    d["target"][3, 6, 4, :] = 0xFF80   # a target row of -inf only
    gt, ga, gb = run_multidraft(d, cfg.temperature)
    assert svpkg.get_status() == -4
    assert svpkg.get_status() == 0
    assert (ga[:4] == -1).all() and (gt[:4] == -1).all() and (gb[:4] == -1).all()
    compare_multidraft(d, cfg.temperature, gpu=(gt, ga, gb))
