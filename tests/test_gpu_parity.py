"""GPU parity: libspecverify (through its C ABI) against the CPU oracle.

Sampling mode: tokens and accept lengths identical except at near-ties
(|u - alpha|, CDF gap / Z or top-p cumulative gap below 1e-6, counted);
normalisers within 1e-5. Greedy mode: bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg
from gpu_util import compare_greedy, compare_row_stats, compare_sample, run_sample, to_dev

pytestmark = pytest.mark.gpu

C = sg.CONFIGS


@pytest.fixture(scope="module", autouse=True)
def built():
    svpkg.build()
    torch.cuda.set_device(0)
    svpkg.set_launch_shape(0, 0)
    yield
    assert svpkg.get_status() == 0


SAMPLE_CASES = {
    "cfg1_b300": C["cfg1_v1000_f32"].with_(B=300),
    "cfg2_b16": C["cfg2_v32000_bf16"].with_(B=16),
    "cfg3_b6": C["cfg3_v128256_bf16"].with_(B=6),
    "cfg5_b6_topp": C["cfg5_topp_v151936_bf16"].with_(B=6),
    "ragged_bf16_v32007": C["cfg2_v32000_bf16"].with_(B=8, K=3, V=32007),
    "ragged_f32_v1001": C["cfg1_v1000_f32"].with_(B=64, V=1001),
    "tiny_v2": C["cfg1_v1000_f32"].with_(B=400, K=2, V=2),
    "tiny_v3_bf16": C["cfg2_v32000_bf16"].with_(B=400, K=2, V=3),
    "v17_k1": C["cfg2_v32000_bf16"].with_(B=300, K=1, V=17),
    "topp_f32": C["cfg1_v1000_f32"].with_(B=40, V=5000, temperature=0.5, top_p=0.5),
    "topp_ragged_bf16": C["cfg5_topp_v151936_bf16"].with_(B=6, K=3, V=20011, top_p=0.8),
    "topp_flat": C["cfg2_v32000_bf16"].with_(B=6, K=2, V=9000, target_sigma=0.05, draft_sigma=0.02, top_p=0.95,
                                             n_peaks=0),
    # top-p decide: clusters of 2, 4 and 16 CTAs per sequence; a flat row
    # whose cut lies below the row pass's first window of keys (and whose
    # nucleus spans the row); a nucleus of about one token
    "topp_d2_v40000": C["cfg5_topp_v151936_bf16"].with_(B=6, K=3, V=40000),
    "topp_d4_flat_v70000": C["cfg2_v32000_bf16"].with_(B=4, K=2, V=70000, target_sigma=0.05, draft_sigma=0.02,
                                                       top_p=0.95, n_peaks=0),
    "topp_d16_v200000": C["cfg5_topp_v151936_bf16"].with_(B=2, K=2, V=200000),
    "topp_p005_v32000": C["cfg5_topp_v151936_bf16"].with_(B=8, K=4, V=32000, top_p=0.05),
    "hot_T2": C["cfg2_v32000_bf16"].with_(B=10, K=4, V=16384, temperature=2.0),
    # whole sequences in one CTA (2K+1 rows within 48 KB, rows 16-byte aligned);
    # rows of at most 1024 elements: one warp per sequence
    "seqmode_bf16_v2048_k3": C["cfg2_v32000_bf16"].with_(B=50, K=3, V=2048),
    "seqmode_f32_v8_k2": C["cfg1_v1000_f32"].with_(B=400, K=2, V=8),
    "seqmode_bf16_v512_k15": C["cfg2_v32000_bf16"].with_(B=40, K=15, V=512, temperature=0.6),
    "warpmode_f32_v1024_k7": C["cfg1_v1000_f32"].with_(B=700, K=7, V=1024),
    "warpmode_bf16_v16_k31": C["cfg2_v32000_bf16"].with_(B=90, K=31, V=16, temperature=1.3),
}


@pytest.mark.parametrize("path", [2, 1])
@pytest.mark.parametrize("name", sorted(SAMPLE_CASES))
def test_sample_parity(name, path):
    # path 2: the row pass and the cluster decide kernel wherever they fit;
    # path 1: the streaming kernel
    cfg = SAMPLE_CASES[name]
    d = sg.sample_inputs(cfg)
    svpkg.set_sample_path(path)
    try:
        gpu = run_sample(d, cfg.temperature, cfg.top_p, row_stats=True)
    finally:
        svpkg.set_sample_path(0)
    compare_sample(d, cfg.temperature, cfg.top_p, gpu=gpu, max_mismatch=1)
    compare_row_stats(d, gpu[2], cfg.temperature, cfg.top_p)


GREEDY_CASES = {
    "cfg4_b4": C["cfg4_greedy_v32000_bf16"].with_(B=4),
    "ragged_v32007": C["cfg4_greedy_v32000_bf16"].with_(B=3, V=32007),
    "f32_v1001": C["cfg4_greedy_v32000_bf16"].with_(B=20, V=1001, dtype=sg.F32),
    "g1_n2": C["cfg4_greedy_v32000_bf16"].with_(B=50, G=1, N=2, V=300),
    "many_cand": C["cfg4_greedy_v32000_bf16"].with_(B=5, G=40, N=9, V=2000),
}


@pytest.mark.parametrize("name", sorted(GREEDY_CASES))
def test_greedy_parity(name):
    compare_greedy(sg.greedy_inputs(GREEDY_CASES[name]))


def test_greedy_ties_lowest_index():
    # logits on a coarse grid: many equal maxima, including -0 against +0
    cfg = C["cfg4_greedy_v32000_bf16"].with_(B=30, V=3000)
    d = sg.greedy_inputs(cfg)
    x = np.round(sg.to_float(d["logits"], sg.BF16) / 4.0)
    x[x == 0] = -0.0
    x[..., ::7][x[..., ::7] == -0.0] = 0.0
    d["logits"] = sg.from_float(x, sg.BF16)
    # keep the candidates' prefix structure meaningful under the new argmax
    a = x.argmax(-1)
    d["cand"][:, :, :2] = a[:, :, :2]
    compare_greedy(d)


def test_greedy_limit_of_sampling():
    cfg = C["cfg2_v32000_bf16"].with_(B=40, V=3001, temperature=0.0)
    d = sg.sample_inputs(cfg)
    gt, ga = svpkg.verify_sample(to_dev(d["target"]), None, to_dev(d["draft_tokens"]), None, 0.0)
    rt, ra, _ = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 0.0)
    np.testing.assert_array_equal(ga.cpu().numpy(), ra)
    np.testing.assert_array_equal(gt.cpu().numpy(), rt)


def test_identical_models_accept_everything():
    cfg = C["cfg2_v32000_bf16"].with_(B=20, K=6, V=5000)
    d = sg.sample_inputs(cfg)
    d["draft"] = np.ascontiguousarray(d["target"][:, : cfg.K])
    d["draft_tokens"] = sg.draft_tokens(d["draft"], cfg.dtype, cfg.temperature, cfg.top_p, seed=4)
    gt, ga = run_sample(d, cfg.temperature)
    assert (ga == cfg.K).all()
    compare_sample(d, cfg.temperature, gpu=(gt, ga))


def test_disjoint_supports_reject_first():
    cfg = C["cfg1_v1000_f32"].with_(B=64, K=3, V=64)
    d = sg.sample_inputs(cfg)
    t = d["target"].copy()
    dr = d["draft"].copy()
    t[:, :, 32:] = -np.inf
    dr[:, :, :32] = -np.inf
    d["target"], d["draft"] = t, dr
    d["draft_tokens"] = sg.draft_tokens(dr, cfg.dtype, cfg.temperature, seed=9)
    gt, ga = run_sample(d, cfg.temperature)
    assert (ga == 0).all() and (gt[:, 0] < 32).all()
    compare_sample(d, cfg.temperature, gpu=(gt, ga))


def test_bad_inputs_flag_only_their_sequence():
    cfg = C["cfg2_v32000_bf16"].with_(B=8, K=3, V=4000)
    d = sg.sample_inputs(cfg)
    d["draft_tokens"][0, 1] = cfg.V
    d["draft_tokens"][1, 0] = -5
    d["uniforms"][2, 3] = 1.0
    d["target"][3, 2, 17] = 0x7FC0   # NaN
    d["draft"][4, 1, 9] = 0x7F80     # +inf
    d["target"][5, 0, :] = 0xFF80    # all -inf
    gt, ga = run_sample(d, cfg.temperature)
    assert svpkg.get_status() == -4
    assert svpkg.get_status() == 0  # the flag is cleared by reading it
    assert (ga[:6] == -1).all() and (gt[:6] == -1).all()
    rt, ra, _ = oracle.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], cfg.temperature)
    np.testing.assert_array_equal(ra[:6], -1)
    compare_sample(d, cfg.temperature, gpu=(gt, ga))
    g = sg.greedy_inputs(C["cfg4_greedy_v32000_bf16"].with_(B=3, V=500))
    g["cand"][1, 2, 1] = 500
    g["logits"][2, 0, 0, 3] = 0x7FC0
    compare_greedy(g)
    assert svpkg.get_status() == -4


@pytest.mark.parametrize("V", [1024, 2048])  # one warp per sequence / one CTA per sequence
def test_bad_inputs_in_sequence_mode(V):
    cfg = C["cfg2_v32000_bf16"].with_(B=8, K=3, V=V)
    d = sg.sample_inputs(cfg)
    d["draft_tokens"][0, 1] = cfg.V
    d["uniforms"][2, 3] = 1.0
    d["target"][3, 2, 17] = 0x7FC0   # NaN
    d["draft"][4, 1, 9] = 0x7F80     # +inf
    d["target"][5, 0, :] = 0xFF80    # all -inf
    gt, ga = run_sample(d, cfg.temperature)
    assert svpkg.get_status() == -4
    assert (ga[[0, 2, 3, 4, 5]] == -1).all() and (ga[[1, 6, 7]] >= 0).all()
    compare_sample(d, cfg.temperature, gpu=(gt, ga))


def test_bounded_wait_reports_timeout_and_recovers():
    # A wait that nothing ends gives up after its limit (10 ms here) and
    # reports SV_ERR_TIMEOUT; the stream's scratch is reset and later calls work.
    assert svpkg.get_status() == 0
    svpkg.selftest_wait_timeout(10_000_000)
    assert svpkg.get_status() == -5
    assert svpkg.get_status() == 0
    cfg = C["cfg2_v32000_bf16"].with_(B=6, V=9000)
    d = sg.sample_inputs(cfg)
    compare_sample(d, cfg.temperature, max_mismatch=1)
    assert svpkg.get_status() == 0


def test_empty_batch_is_a_noop():
    e = torch.empty((0, 5, 100), dtype=torch.bfloat16, device="cuda")
    ot, oa = svpkg.verify_sample(e, torch.empty((0, 4, 100), dtype=torch.bfloat16, device="cuda"),
                                 torch.empty((0, 4), dtype=torch.int32, device="cuda"),
                                 torch.empty((0, 5), dtype=torch.float32, device="cuda"), 1.0)
    assert ot.shape == (0, 5) and oa.shape == (0,)


def test_host_buffers_match_device_path():
    cfg = C["cfg2_v32000_bf16"].with_(B=12, V=7000)
    d = sg.sample_inputs(cfg)
    dev = run_sample(d, cfg.temperature)

    def host(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
        return torch.from_numpy(a).pin_memory()

    ht, ha = svpkg.verify_sample(host(d["target"]), host(d["draft"]), host(d["draft_tokens"]), host(d["uniforms"]),
                                 cfg.temperature)
    assert ht.device.type == "cpu"
    np.testing.assert_array_equal(ht.numpy(), dev[0])
    np.testing.assert_array_equal(ha.numpy(), dev[1])


def test_repeatable_and_stream_local():
    cfg = C["cfg3_v128256_bf16"].with_(B=5, V=50000)
    d = sg.sample_inputs(cfg)
    a = run_sample(d, cfg.temperature)
    b = run_sample(d, cfg.temperature)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    args = [to_dev(d[k]) for k in ("target", "draft", "draft_tokens", "uniforms")]
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        r1 = svpkg.verify_sample(*args, cfg.temperature)
    with torch.cuda.stream(s2):
        r2 = svpkg.verify_sample(*args, cfg.temperature)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(r1[0].cpu().numpy(), a[0])
    np.testing.assert_array_equal(r2[0].cpu().numpy(), a[0])
    np.testing.assert_array_equal(r1[1].cpu().numpy(), a[1])
    np.testing.assert_array_equal(r2[1].cpu().numpy(), a[1])


@pytest.mark.parametrize("stages,ctas", [(1, 1), (2, 3), (4, 1), (6, 1)])
def test_launch_shapes_agree(stages, ctas):
    cfg = C["cfg5_topp_v151936_bf16"].with_(B=4, V=40000)
    d = sg.sample_inputs(cfg)
    ref = run_sample(d, cfg.temperature, cfg.top_p)
    try:
        svpkg.set_launch_shape(stages, ctas)
        got = run_sample(d, cfg.temperature, cfg.top_p)
        g = sg.greedy_inputs(C["cfg4_greedy_v32000_bf16"].with_(B=2, V=9000))
        compare_greedy(g)
    finally:
        svpkg.set_launch_shape(0, 0)
    for x, y in zip(ref, got):
        np.testing.assert_array_equal(x, y)


# ------------------------------------------------------------------ full size
# The measured workloads at their full sizes, in the launch configuration the
# benchmark times; every sequence is checked against the oracle.

@pytest.mark.parametrize("name", ["cfg1_v1000_f32", "cfg2_v32000_bf16", "cfg3_v128256_bf16",
                                  "cfg5_topp_v151936_bf16"])
def test_full_size_sample(name):
    cfg = C[name]
    d = sg.sample_inputs(cfg)
    gpu = run_sample(d, cfg.temperature, cfg.top_p, row_stats=True)
    summary = compare_sample(d, cfg.temperature, cfg.top_p, gpu=gpu, max_mismatch=1)
    rows = np.random.default_rng(0).choice(cfg.rows, size=min(cfg.rows, 48), replace=False)
    compare_row_stats(d, gpu[2], cfg.temperature, cfg.top_p, rows=rows)
    print(name, summary)


def test_full_size_greedy():
    s = compare_greedy(sg.greedy_inputs(C["cfg4_greedy_v32000_bf16"]))
    print("cfg4", s)


def test_alternating_shapes_on_one_stream():
    # calls of different shapes and modes reuse one scratch area: every call
    # must start from clean counters whatever ran before it
    cases = [sg.sample_inputs(C["cfg2_v32000_bf16"].with_(B=9, V=3001)),
             sg.greedy_inputs(C["cfg4_greedy_v32000_bf16"].with_(B=5, V=777, dtype=sg.F32)),
             sg.sample_inputs(C["cfg1_v1000_f32"].with_(B=70, K=2, V=129)),
             sg.greedy_inputs(C["cfg4_greedy_v32000_bf16"].with_(B=2, G=3, N=3, V=20000))]
    for _ in range(2):
        for d in cases:
            if "logits" in d:
                compare_greedy(d)
            else:
                temp = 1.0
                compare_sample(d, temp)


@pytest.mark.parametrize("path", [0, 1])
def test_greedy_paths_agree(path):
    # the streaming kernel and the row-argmax + match kernels, bit-exact
    svpkg.set_greedy_path(path)
    try:
        for cfg in (C["cfg4_greedy_v32000_bf16"], C["cfg4_greedy_v32000_bf16"].with_(B=9, V=1001, dtype=sg.F32),
                    C["cfg4_greedy_v32000_bf16"].with_(B=5, G=40, N=3, V=333)):
            compare_greedy(sg.greedy_inputs(cfg))
        g = sg.greedy_inputs(C["cfg4_greedy_v32000_bf16"].with_(B=3, V=500))
        g["cand"][1, 2, 1] = 500
        g["logits"][2, 0, 0, 3] = 0x7FC0
        compare_greedy(g)
        assert svpkg.get_status() == -4
    finally:
        svpkg.set_greedy_path(0)
