"""The benchmark's host side, without a GPU: the algorithmic bytes and
positions it credits per call, and the JSON line of its reference arm (the
CPU oracle on a bounded sample)."""
import json
import os
import subprocess
import sys

import pytest

import bench
import specgen as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", list(sg.CONFIGS) + list(sg.LOOKAHEAD_CONFIGS) + list(sg.MULTIDRAFT_CONFIGS))
def test_algorithmic_bytes_are_one_read_of_every_logit(name):
    cfg, mode, positions, logit_bytes, small_in, out_bytes = bench.workload(name)
    s = 2 if cfg.dtype == sg.BF16 else 4
    if mode == "multidraft":
        assert positions == cfg.B * cfg.G * cfg.N
        assert logit_bytes == cfg.B * cfg.G * (2 * cfg.N - 1) * cfg.V * s
    elif mode == "sample":
        assert positions == cfg.B * (cfg.K + 1)
        assert logit_bytes == cfg.B * (2 * cfg.K + 1) * cfg.V * s
        assert out_bytes == cfg.B * (cfg.K + 1) * 4 + cfg.B * 4
    else:
        assert positions == cfg.B * cfg.G * cfg.N
        assert logit_bytes == cfg.B * cfg.G * cfg.N * cfg.V * s
        assert out_bytes == cfg.B * cfg.N * 4 + cfg.B * 4
    assert mode == {"cfg4_greedy_v32000_bf16": "greedy", "la_sample_v32000_bf16": "lookahead",
                    "md_sample_v32000_bf16": "multidraft"}.get(name, "sample")
    c = bench.config_json(cfg, mode, 3)
    assert c["workload"] == name and c["B"] == cfg.B and c["V"] == cfg.V


def test_batch_override_names_the_workload():
    cfg, mode, *_ = bench.workload("cfg1_v1000_f32", batch=1)
    assert cfg.B == 1 and bench.config_json(cfg, mode, 1)["workload"] == "cfg1_v1000_f32_b1"


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config",
                        "cfg1_v1000_f32", "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3 and line["config"]["workload"] == "cfg1_v1000_f32"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_config_names():
    assert bench.config_names("cfg2_v32000_bf16") == ["cfg2_v32000_bf16"]
    assert bench.config_names("cfg1_v1000_f32, la_sample_v32000_bf16") == ["cfg1_v1000_f32", "la_sample_v32000_bf16"]
    every = (list(sg.CONFIGS) + list(sg.LOOKAHEAD_CONFIGS) + list(sg.MULTIDRAFT_CONFIGS) +
             list(bench.POOL_WORKLOADS) + list(bench.LMHEAD_WORKLOADS))
    # the headline workload (the largest) first, then every other one, each once
    for spec in ("all", None):
        names = bench.config_names(spec)
        assert names[0] == "cfg3_v128256_bf16" and sorted(names) == sorted(every)
    with pytest.raises(KeyError):
        bench.config_names("cfg2_v32000_bf16,nope")
    # the pool and the LM-head verify are per_config records (or --calls targets)
    assert bench.config_names("cfg2_v32000_bf16,ngram_pool_v32000,lmhead_d4096_v32000") == [
        "cfg2_v32000_bf16", "ngram_pool_v32000", "lmhead_d4096_v32000"]
    assert bench.config_names("ngram_pool_v32000") == ["ngram_pool_v32000"]


def test_pool_inputs_are_seeded_and_hit_the_keys():
    w = bench.POOL_WORKLOADS["ngram_pool_v32000"]
    a, la = bench.pool_inputs(w, 4)
    b, lb = bench.pool_inputs(w, 4)
    assert (a == b).all() and (la == lb).all()
    assert a.shape == (4, w["B"], w["W"], w["N"]) and la.shape == (4, w["B"])
    assert a[..., 0].max() < w["keys"] and la.max() < w["keys"] and a.max() < w["V"] and a.min() >= 0


def test_launched_kernel_follows_the_library_rule():
    class A:
        sample_path = 0
        greedy_path = 0
    for name, kernel in (("cfg1_v1000_f32", "verify_warp_kernel"), ("cfg3_v128256_bf16", "verify_kernel"),
                         ("cfg2_v32000_bf16", "rows_kernel"),
                         ("cfg5_topp_v151936_bf16", "topp_rows_kernel"), ("cfg4_greedy_v32000_bf16", "gr_rows_kernel"),
                         ("la_sample_v32000_bf16", "la_rows_kernel"), ("md_sample_v32000_bf16", "md_rows_kernel")):
        cfg, mode = bench.workload(name)[:2]
        assert bench.launched_kernel(cfg, mode, A) == kernel, name
    A.sample_path = A.greedy_path = 1
    cfg, mode = bench.workload("cfg1_v1000_f32")[:2]
    assert bench.launched_kernel(cfg, mode, A) == "verify_warp_kernel"
    cfg, mode = bench.workload("cfg4_greedy_v32000_bf16")[:2]
    assert bench.launched_kernel(cfg, mode, A) == "verify_kernel"


def test_launched_kernel_topp_streaming_on_request():
    class A:
        sample_path = 1
        greedy_path = 0
    cfg, mode = bench.workload("cfg5_topp_v151936_bf16")[:2]
    assert bench.launched_kernel(cfg, mode, A) == "verify_kernel"


def test_every_record_has_current_profiled_traffic():
    # Every workload's streaming kernel (and the pool's and the LM head's
    # kernels) has an ncu summary under profiles/ taken on the sources as they
    # are: a kernel changed since its capture reads as None here.
    class A:
        sample_path = 0
        greedy_path = 0
    for name in list(sg.CONFIGS) + list(sg.LOOKAHEAD_CONFIGS) + list(sg.MULTIDRAFT_CONFIGS):
        cfg, mode = bench.workload(name)[:2]
        kernel = bench.launched_kernel(cfg, mode, A)
        assert bench.profiled_traffic(name, kernel) is not None, (name, kernel)
    assert bench.profiled_traffic("lmhead_d4096_v32000", "lmhead_kernel") is not None
    assert bench.pool_traffic("ngram_pool_v32000") is not None
