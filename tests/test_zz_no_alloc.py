"""sv_verify_sample_noalloc: the sampling-mode verify for callers that cannot
allocate device memory (code inside a memory pool or arena that accounts for
every byte, allocator hooks that must not recurse into cudaMalloc, services
that reserve all device memory at start-up). It runs the same kernels as
sv_verify_sample, chosen by the same rule, on a fixed scratch array inside the
library, so it must give the same results; it is also checked against the
oracle directly. Both entry points are called through the C ABI.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import specgen as sg
import speculative_decoding_verification_39_gb300 as svpkg

pytestmark = pytest.mark.gpu

SV_ERR_SCRATCH_LIMIT = -7


def _dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _call(fn, d, cfg, stream):
    B, K, V = cfg.B, cfg.K, cfg.V
    tokens = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    stats = torch.full((B, 2 * K + 1, 4), float("nan"), dtype=torch.float32, device="cuda")
    rc = fn(_p(d["target"]), _p(d["draft"]), _p(d["draft_tokens"]), _p(d["uniforms"]), B, K, V, cfg.dtype,
            float(cfg.temperature), float(cfg.top_p), _p(tokens), _p(acc), _p(stats), stream)
    assert rc == 0, rc
    return tokens, acc, stats


CASES = {
    # the row pass + cluster decide kernels
    "cfg2_v20011": sg.CONFIGS["cfg2_v32000_bf16"].with_(B=12, V=20011),
    # short fp32 rows (a group of rows per CTA in the row pass)
    "cfg1_v1000_f32": sg.CONFIGS["cfg1_v1000_f32"].with_(B=300),
    # top-p: the streaming kernel
    "cfg5_topp_v20011": sg.CONFIGS["cfg5_topp_v151936_bf16"].with_(B=12, V=20011),
    # T = 0, the greedy limit: the streaming kernel's argmax mode
    "cfg2_greedy_limit": sg.CONFIGS["cfg2_v32000_bf16"].with_(B=12, V=20011, temperature=0.0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_sample_on_two_calls(name):
    svpkg.build()
    lib = svpkg.lib()
    torch.cuda.set_device(0)
    cfg = CASES[name]
    host = sg.sample_inputs(cfg)
    d = {k: _dev(v) for k, v in host.items()}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref = _call(lib.sv_verify_sample, d, cfg, stream)
    first = _call(lib.sv_verify_sample_noalloc, d, cfg, stream)
    second = _call(lib.sv_verify_sample_noalloc, d, cfg, stream)
    torch.cuda.synchronize()
    rt, ra, rs = (x.cpu().numpy() for x in ref)
    assert (ra >= 0).all()
    for got in (first, second):
        gt, ga, gs = (x.cpu().numpy() for x in got)
        np.testing.assert_array_equal(ga, ra)
        np.testing.assert_array_equal(gt, rt)
        np.testing.assert_allclose(gs, rs, rtol=1e-5, atol=1e-5)
    # and against the oracle: identical except at near-ties (margin < 1e-6)
    ot, oa, margin = oracle.verify_sample(host["target"], host["draft"], host["draft_tokens"], host["uniforms"],
                                          cfg.temperature, cfg.top_p)
    gt, ga = second[0].cpu().numpy(), second[1].cpu().numpy()
    diff = (ga != oa) | (gt != ot).any(1)
    assert not (diff & (margin >= 1e-6)).any(), np.nonzero(diff)[0]
    assert diff.sum() <= 1


def test_noalloc_rejects_a_call_beyond_its_scratch():
    svpkg.build()
    lib = svpkg.lib()
    torch.cuda.set_device(0)
    x = torch.zeros(16, dtype=torch.int32, device="cuda")  # never read: the size check comes first
    p = _p(x)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.sv_verify_sample_noalloc(p, p, p, p, 200000, 8, 128256, 1, 1.0, 1.0, p, p, None, stream)
    assert rc == SV_ERR_SCRATCH_LIMIT
    assert lib.sv_status_string(rc) == b"the call needs more than the fixed no-allocation scratch"
