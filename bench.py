#!/usr/bin/env python3
"""Benchmark of the speculative-decoding verify step (libspecverify, GB300).

One step = one verify call over one batch of the workload: every row of
target and draft logits read once, the accept scan, and the residual or bonus
draw. Metric: verified positions per second (B*(K+1) target positions per
sampling call, B*G*N per greedy call), with the achieved algorithmic HBM
bandwidth (one read of every logit) against the measured peak.

Headline workload: B=256, K=8, V=128256 bf16, T=0.8 — the largest of the five
verify workloads and the largest that one GPU holds several copies of. The
same JSON line carries a ``per_config`` record for every other workload (the
four other verify workloads, the Lookahead sampling verify and the multi-draft
verify), each with its own throughput, roofline, end-to-end figure, CPU
baseline and GPU/oracle mismatch counts.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME[,NAME..]|all] [--impl reference]

Timing: inputs are resident in HBM before the timed region; the K timed calls
are replayed from CUDA graphs, cycling through enough copies of the inputs
that the working set exceeds the 129 MB L2 (so no call finds its inputs in
L2); CUDA events on the launching stream bracket the timed replays, with a
barrier and a device synchronise on both sides. That is the pipelined
per-call time: consecutive calls on the stream may overlap their launch and
ramp. ``isolated_us`` is the per-call time with every call followed by a
one-element torch kernel that ends the overlap, minus that kernel's own time.
``e2e`` repeats the metric through the public API with pinned host buffers,
copies included. ``--impl reference`` times the CPU oracle (the baseline this
project is checked against) on a bounded sample of the same workload.

Two more per_config records are not verify calls of logits: the Lookahead
n-gram pool (one insert and one lookup per step) and the verify on LM-head
hidden states (the tcgen05 GEMM h.W^T of both heads, then the verify).

``--calls N`` runs N plain calls of the first named workload (no graphs, no
timing, no oracle) and exits: the command the ncu summaries under profiles/
are taken with.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import specgen as sg  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
DEFAULT_CONFIG = "cfg3_v128256_bf16"
KERNEL = "verify_kernel"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ workload

# The Lookahead n-gram pool ("Lookahead Decoding 完全拆解", "N-gram 池与身份判定"):
# per step, every sequence inserts the W n-grams of one Lookahead window step
# and looks up G candidates for its last token (the greedy workload's shape:
# B = 32, G = W = 7, N = 5, V = 32000; at most cap = 7 n-grams per first
# token). First tokens and last tokens come from 64 ids, so that lookups find
# n-grams; the other tokens are uniform over the vocabulary.
POOL_WORKLOADS = {"ngram_pool_v32000": {"B": 32, "V": 32000, "N": 5, "cap": 7, "G": 7, "W": 7, "keys": 64}}

# The verify on LM-head hidden states (reading c24): cfg2's verify shape
# (B = 64, K = 5, V = 32000, T = 1) on hidden states of D = 4096, the hidden
# size of the 7B models the pages use as targets and drafts; hidden states
# N(0, 1) and heads N(0, 1/D), bf16, seeded.
LMHEAD_WORKLOADS = {"lmhead_d4096_v32000": {"B": 64, "K": 5, "D": 4096, "V": 32000, "T": 1.0}}
EXTRA_WORKLOADS = set(POOL_WORKLOADS) | set(LMHEAD_WORKLOADS)


def find_config(name: str):
    for table in (sg.CONFIGS, sg.LOOKAHEAD_CONFIGS, sg.MULTIDRAFT_CONFIGS):
        if name in table:
            return table[name]
    raise KeyError(name)


def workload(name: str, batch: int | None = None):
    """(cfg, mode, positions, logit bytes, small input bytes, output bytes) of
    one call; mode is "sample", "greedy" or "lookahead" (the sampling-mode
    Lookahead verify)."""
    cfg = find_config(name)
    if batch:
        cfg = cfg.with_(B=batch)
    mode = ("greedy" if isinstance(cfg, sg.GreedyConfig) else
            "lookahead" if isinstance(cfg, sg.LookaheadSampleConfig) else
            "multidraft" if isinstance(cfg, sg.MultiDraftConfig) else "sample")
    esz = 2 if cfg.dtype == sg.BF16 else 4
    if mode == "multidraft":
        positions = cfg.B * cfg.G * cfg.N
        logit_bytes = cfg.B * cfg.G * (2 * cfg.N - 1) * cfg.V * esz
        small_in = cfg.B * cfg.G * (cfg.N - 1) * 4 + cfg.B * ((cfg.N - 1) * cfg.G + 1) * 4
        out_bytes = cfg.B * cfg.N * 4 + cfg.B * 4
    elif mode != "sample":
        positions = cfg.B * cfg.G * cfg.N
        logit_bytes = cfg.B * cfg.G * cfg.N * cfg.V * esz
        small_in = cfg.B * cfg.G * (cfg.N - 1) * 4
        if mode == "lookahead":
            small_in += cfg.B * ((cfg.N - 1) * cfg.G + 1) * 4
        out_bytes = cfg.B * cfg.N * 4 + cfg.B * 4
    else:
        positions = cfg.B * (cfg.K + 1)
        logit_bytes = cfg.B * (2 * cfg.K + 1) * cfg.V * esz
        small_in = cfg.B * cfg.K * 4 + cfg.B * (cfg.K + 1) * 4
        out_bytes = cfg.B * (cfg.K + 1) * 4 + cfg.B * 4
    return cfg, mode, positions, logit_bytes, small_in, out_bytes


def kernel_for(cfg, mode) -> str:
    """Which kernel the library launches for this workload (the library's own
    selection rule, restated for the report): one warp per sequence for rows of
    at most 1024 elements, one CTA per sequence when a whole sequence fits
    48 KB, else the streaming kernel. Inputs here are always 16-byte aligned.
    The Lookahead sampling verify streams its rows in la_rows_kernel."""
    if mode == "lookahead":
        return "la_rows_kernel"
    if mode == "multidraft":
        return "md_rows_kernel"
    if mode == "greedy" or cfg.temperature == 0.0 or cfg.top_p < 1.0:
        return KERNEL
    esz = 2 if cfg.dtype == sg.BF16 else 4
    rows = 2 * cfg.K + 1
    if (cfg.V * esz) % 16 != 0 or rows > 64:
        return KERNEL
    if cfg.V <= 1024 and rows * cfg.V * esz <= 65536:
        return "verify_warp_kernel"
    if rows * cfg.V * esz <= 49152:
        return "verify_seq_kernel"
    return KERNEL


def config_json(cfg, mode, rotation, l2_resident=False):
    c = {"workload": cfg.name if cfg.B == find_config(cfg.name).B else f"{cfg.name}_b{cfg.B}", "B": cfg.B,
         "V": cfg.V, "logits": "bf16" if cfg.dtype == sg.BF16 else "f32"}
    if mode == "greedy":
        c.update({"mode": "greedy", "G": cfg.G, "N": cfg.N})
    elif mode == "lookahead":
        c.update({"mode": "lookahead_sample", "G": cfg.G, "N": cfg.N, "temperature": cfg.temperature})
    elif mode == "multidraft":
        c.update({"mode": "multidraft_sample", "G": cfg.G, "N": cfg.N, "temperature": cfg.temperature})
    else:
        c.update({"mode": "sample", "K": cfg.K, "temperature": cfg.temperature, "top_p": cfg.top_p})
    esz = 2 if cfg.dtype == sg.BF16 else 4
    fits = workload(cfg.name, cfg.B)[3] <= L2_BYTES
    if l2_resident and fits:
        c["l2"] = "L2-resident: one input set replayed (not an HBM figure)"
    else:
        c["l2"] = (f"inputs larger than L2: {rotation} rotating input sets" if rotation > 1
                   else "inputs larger than L2 (one set)")
    return c


def to_torch(a, torch, pin=False):
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
    return t.pin_memory() if pin else t


# -------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources each kernel is built from: a profiled traffic figure is only
# reported while they are the ones that were profiled.
KERNEL_SOURCES = {
    "rows_kernel": ("sv_rows.cu", "sv_v2.h", "sv_device.cuh"),
    "topp_rows_kernel": ("sv_rows.cu", "sv_v2.h", "sv_device.cuh"),
    "refine_kernel": ("sv_refine.cu", "sv_refine.h", "sv_df.cuh", "sv_device.cuh"),
    "decide_kernel": ("sv_decide.cu", "sv_df.cuh", "sv_v2.h", "sv_refine.h", "sv_device.cuh"),
    "verify_kernel": ("sv_kernels.cu", "sv_device.cuh", "sv_kernels.h"),
    "verify_warp_kernel": ("sv_kernels.cu", "sv_device.cuh", "sv_kernels.h"),
    "verify_seq_kernel": ("sv_kernels.cu", "sv_device.cuh", "sv_kernels.h"),
    "gr_rows_kernel": ("sv_greedy_rows.cu", "sv_greedy_rows.h", "sv_device.cuh"),
    "la_rows_kernel": ("sv_lookahead.cu", "sv_lookahead.h", "sv_device.cuh"),
    "md_rows_kernel": ("sv_multidraft.cu", "sv_multidraft.h", "sv_rowstat.cuh", "sv_device.cuh"),
    "md_walk_res_kernel": ("sv_multidraft.cu", "sv_multidraft.h", "sv_rowstat.cuh", "sv_device.cuh"),
    "gr_match_kernel": ("sv_greedy_rows.cu", "sv_greedy_rows.h", "sv_device.cuh"),
    "la_walk_kernel": ("sv_lookahead.cu", "sv_lookahead.h", "sv_device.cuh"),
    "insert_staged_kernel": ("sv_ngram.cu", "sv_device.cuh", "sv_sample_impl.h"),
    "lookup_kernel": ("sv_ngram.cu", "sv_device.cuh", "sv_sample_impl.h"),
    "lmhead_kernel": ("sv_lmhead.cu", "sv_lmhead.h", "sv_device.cuh"),
}


def kernel_source_hash(kernel: str = "verify_kernel") -> str:
    """Hash of the sources of ``kernel``."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_39_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str, kernel: str = "verify_kernel"):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary of
    this workload (profiles/<kernel>_<workload>.md), or None if there is none
    or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload_name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not h or kernel not in KERNEL_SOURCES or h.group(1) != kernel_source_hash(kernel):
        return None
    return float(m.group(1))


def pool_traffic(workload_name: str):
    """DRAM bytes of one pool step (its insert and its lookup launch) from the
    two committed ncu summaries, or None if either is missing or stale."""
    a = profiled_traffic(workload_name, "insert_staged_kernel")
    b = profiled_traffic(workload_name, "lookup_kernel")
    return None if a is None or b is None else a + b


def launched_kernel(cfg, mode, args) -> str:
    """The streaming kernel (the one that reads the logits) the library
    launches for this workload, by the library's own selection rule."""
    if mode == "greedy":
        return "gr_rows_kernel" if args.greedy_path == 0 else "verify_kernel"
    if mode == "lookahead":
        return "la_rows_kernel"
    if mode == "multidraft":
        return "md_rows_kernel"
    esz = 2 if cfg.dtype == sg.BF16 else 4
    small = cfg.B * (2 * cfg.K + 1) * cfg.V * esz <= 96 * 1024 * 1024
    rows = 2 * cfg.K + 1
    warp_rows = cfg.V <= 1024 and (cfg.V * esz) % 16 == 0 and rows <= 64 and rows * cfg.V * esz <= 65536
    if (cfg.temperature > 0 and cfg.top_p < 1.0 and args.sample_path != 1 and esz == 2 and cfg.V % 8 == 0
            and cfg.V <= 327680 and cfg.K <= 1024):
        return "topp_rows_kernel"
    if (cfg.temperature > 0 and cfg.top_p == 1.0 and cfg.K <= 1024 and cfg.V <= 1048576
            and (args.sample_path == 2 or (args.sample_path == 0 and small and not warp_rows))):
        return "rows_kernel"
    if args.sample_path == 0 and cfg.temperature > 0 and cfg.top_p == 1.0 and not warp_rows:
        return KERNEL
    return kernel_for(cfg, mode)


def shard_offset(rank: int, batch: int) -> int:
    """First global sequence of a rank's shard: every rank verifies its own
    ``batch`` sequences of the global batch (weak scaling, no collective)."""
    return rank * batch


def max_over_ranks(value: float, device=None) -> float:
    """The largest of the ranks' values (the timed region's duration)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_inputs(cfg, mode, seq_offset: int = 0, B: int | None = None) -> dict:
    if mode == "greedy":
        return sg.greedy_inputs(cfg, seq_offset=seq_offset, B=B)
    if mode == "lookahead":
        return sg.lookahead_sample_inputs(cfg, seq_offset=seq_offset, B=B)
    if mode == "multidraft":
        return sg.multidraft_inputs(cfg, seq_offset=seq_offset, B=B)
    return sg.sample_inputs(cfg, seq_offset=seq_offset, B=B)


def oracle_cpu_rate(cfg, mode, budget_s: float, nthreads: int):
    """Positions per second of the CPU oracle over a bounded sample of the
    workload, fanned out over sequences on ``nthreads`` host threads."""
    import oracle
    chunk = max(1, min(cfg.B, 8 if cfg.V > 50000 else 32))
    inputs = host_inputs(cfg, mode, B=chunk * nthreads)
    oracle._lib()

    def one(i):
        sl = slice(i * chunk, (i + 1) * chunk)
        if mode == "greedy":
            oracle.verify_greedy(inputs["logits"][sl], inputs["cand"][sl])
        elif mode == "lookahead":
            oracle.verify_lookahead_sample(inputs["logits"][sl], inputs["cand"][sl], inputs["uniforms"][sl],
                                           cfg.temperature)
        elif mode == "multidraft":
            oracle.verify_multidraft_sample(inputs["target"][sl], inputs["draft"][sl], inputs["draft_tokens"][sl],
                                            inputs["uniforms"][sl], cfg.temperature)
        else:
            oracle.verify_sample(inputs["target"][sl], inputs["draft"][sl], inputs["draft_tokens"][sl],
                                 inputs["uniforms"][sl], cfg.temperature, cfg.top_p)
        return chunk

    per_seq = cfg.K + 1 if mode == "sample" else cfg.G * cfg.N
    done, t0 = 0, time.perf_counter()
    with ThreadPoolExecutor(nthreads) as ex:
        while True:
            done += sum(ex.map(one, range(nthreads)))
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    return done * per_seq / el, done, el


# --------------------------------------------------------------- GPU arm

def oracle_counts(host, cfg, mode, gpu_tokens, gpu_acc, nthreads: int):
    """GPU/oracle comparison on one full input set: sequences whose tokens or
    accept length differ, near-ties (the oracle's smallest decision margin
    below 1e-6) and decisions (accept tests and draws; greedy: one per
    sequence). The oracle runs over the sequences on host threads."""
    import oracle
    B = cfg.B
    chunk = max(1, min(32, (B + nthreads - 1) // nthreads))
    sl = [slice(i, min(B, i + chunk)) for i in range(0, B, chunk)]

    def one(s):
        if mode == "greedy":
            t, a, _ = oracle.verify_greedy(host["logits"][s], host["cand"][s])
            return t, a, np.full(len(a), np.inf)
        if mode == "lookahead":
            t, a, _, m = oracle.verify_lookahead_sample(host["logits"][s], host["cand"][s], host["uniforms"][s],
                                                        cfg.temperature)
            return t, a, m
        if mode == "multidraft":
            t, a, _, m = oracle.verify_multidraft_sample(host["target"][s], host["draft"][s],
                                                         host["draft_tokens"][s], host["uniforms"][s],
                                                         cfg.temperature)
            return t, a, m
        return oracle.verify_sample(host["target"][s], host["draft"][s], host["draft_tokens"][s],
                                    host["uniforms"][s], cfg.temperature, cfg.top_p)

    with ThreadPoolExecutor(nthreads) as ex:
        parts = list(ex.map(one, sl))
    rt = np.concatenate([x[0] for x in parts])
    ra = np.concatenate([x[1] for x in parts])
    margin = np.concatenate([x[2] for x in parts])
    diff = (gpu_acc != ra) | (gpu_tokens != rt).any(1)
    near = margin < 1e-6
    if mode == "sample":
        decisions = int(np.where(ra >= 0, np.minimum(ra + 1, cfg.K) + 1, 0).sum())
    elif mode == "greedy":
        decisions = int(B)
    else:
        decisions = int(np.where(ra >= 0, ra + 1, 0).sum())
    return {"sequences": int(B), "decisions": decisions, "mismatch": int(diff.sum()),
            "mismatch_away_from_near_tie": int((diff & ~near).sum()), "near_ties": int(near.sum())}


def measure(args, name: str, rank: int, world: int, steps: int, cpu_budget: float, counts: bool):
    """Times one workload on this rank's GPU; returns its record."""
    import torch
    import speculative_decoding_verification_39_gb300 as svpkg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    cfg, mode, positions, logit_bytes, small_in, out_bytes = workload(name, args.batch)
    rotation = 1 if logit_bytes > L2_BYTES else int(math.ceil(3 * L2_BYTES / logit_bytes)) + 1
    if args.l2_resident:
        rotation = 1  # one input set, replayed: it stays in L2 when it fits
    log(f"[bench] {name}: {logit_bytes / 1e6:.1f} MB of logits per call, {rotation} input set(s)")
    t0 = time.perf_counter()
    off = shard_offset(rank, cfg.B)
    host = host_inputs(cfg, mode, seq_offset=off)
    log(f"[bench] inputs generated in {time.perf_counter() - t0:.1f} s")
    keys = {"greedy": ("logits", "cand"), "lookahead": ("logits", "cand", "uniforms"),
            "multidraft": ("target", "draft", "draft_tokens", "uniforms"),
            "sample": ("target", "draft", "draft_tokens", "uniforms")}[mode]
    pinned = {k: to_torch(host[k], torch, pin=True) for k in keys}
    sets = [{k: pinned[k].to(dev, non_blocking=True) for k in keys} for _ in range(rotation)]
    torch.cuda.synchronize()
    width = cfg.K + 1 if mode == "sample" else cfg.N
    outs = [(torch.empty((cfg.B, width), dtype=torch.int32, device=dev),
             torch.empty((cfg.B,), dtype=torch.int32, device=dev)) for _ in range(rotation)]

    def public_call(*a, **kw):
        if mode == "greedy":
            return svpkg.verify_greedy(*a, **kw)
        if mode == "lookahead":
            return svpkg.verify_lookahead_sample(*a, cfg.temperature, **kw)
        if mode == "multidraft":
            return svpkg.verify_multidraft_sample(*a, cfg.temperature, **kw)
        return svpkg.verify_sample(*a, cfg.temperature, cfg.top_p, **kw)

    def call(i):
        s, (ot, oa) = sets[i % rotation], outs[i % rotation]
        public_call(*(s[k] for k in keys), out_tokens=ot, out_accept_len=oa)

    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            call(i)
    stream.synchronize()
    with torch.cuda.stream(stream):
        if svpkg.get_status() != 0:
            raise RuntimeError("device status set during warm-up")
    breaker = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        refined0 = svpkg.refined_draws()

    def capture(n, idx0, with_breaker=False, only_breaker=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n):
                if not only_breaker:
                    call(idx0 + k)
                if with_breaker or only_breaker:
                    breaker.add_(1)
        return g

    # graphs of at most 1000 calls; the timed region replays exactly `steps` calls
    graphs, n_left, idx = [], steps, 0
    launches_before = svpkg.launch_count()
    while n_left > 0:
        n = min(1000, n_left)
        graphs.append(capture(n, idx))
        idx += n
        n_left -= n
    captured = svpkg.launch_count() - launches_before
    n_iso = 100
    g_iso = capture(n_iso, 0, with_breaker=True)
    g_brk = capture(n_iso, 0, only_breaker=True)

    def timed(gs):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for g in gs:
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    # pre-roll: replay for ~1 s so that clocks settle and the sampler sees the load
    with ClockSampler(local) as clk:
        t_pre = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - t_pre < 1.0:
                graphs[0].replay()
                stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ms = timed(graphs)
        if world > 1:
            torch.distributed.barrier()
        ms_iso = min(timed([g_iso]) for _ in range(3))
        ms_brk = min(timed([g_brk]) for _ in range(3))
    with torch.cuda.stream(stream):
        status = svpkg.get_status()
        refined = svpkg.refined_draws() - refined0
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    ms = max_over_ranks(ms, dev)
    ms_per_step = ms / steps
    iso_us = max(0.0, (ms_iso - ms_brk) / n_iso * 1e3)
    value = positions * world * steps / (ms / 1e3)
    achieved_gbs = logit_bytes / (ms_per_step / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    gt, ga = outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy()

    # end to end through the public API with pinned host buffers
    e2e_steps = max(3, min(20, steps))
    host_args = [pinned[k] for k in keys]
    with torch.cuda.stream(stream):
        for _ in range(2):
            public_call(*host_args)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        for _ in range(e2e_steps):
            public_call(*host_args)
        e2e_s = (time.perf_counter() - t1) / e2e_steps
    h2d = logit_bytes + small_in
    kernel = launched_kernel(cfg, mode, args)
    rec = {
        "workload": config_json(cfg, mode, rotation, args.l2_resident),
        "value": value,
        "unit": "positions/s",
        "ms_per_step": ms_per_step,
        "steps": steps,
        "rounds_per_s": cfg.B * world / (ms_per_step / 1e3),
        "isolated_us": iso_us,
        "isolated_note": f"{n_iso} calls each followed by a one-element torch kernel that ends the launch "
                         f"overlap, minus {n_iso} such kernels alone ({ms_brk * 1e3 / n_iso:.2f} us each)",
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": profiled_traffic(name, kernel), "algorithmic_bytes_per_launch": logit_bytes,
                     "kernel": kernel,
                     "isolated_frac": (logit_bytes / (iso_us * 1e-6) / 1e9 / peak) if iso_us > 0 else None,
                     "timing": "CUDA events over graph replays of the timed calls"},
        "clocks": clk.summary(),
        "e2e": {"value": positions * world / e2e_s, "unit": "positions/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": out_bytes},
        "gpu_launches": int(captured),
        "refined_draws_per_call": refined / max(1, steps + 2 * n_iso + 50),
        "refined_note": "draws redone in double-float because the fp32 walk landed within 1e-7*Z of a CDF edge, "
                        "per call, over every call of the timed graphs and the isolated runs (the pre-roll "
                        "replays are counted too, so this is an estimate)",
    }
    nth = os.cpu_count() or 1
    if counts and rank == 0:
        t2 = time.perf_counter()
        rec["parity"] = oracle_counts(host, cfg, mode, gt, ga, nth)
        log(f"[bench] oracle comparison in {time.perf_counter() - t2:.1f} s: {rec['parity']}")
    if cpu_budget > 0 and rank == 0 and world == 1:
        rate, n, el = oracle_cpu_rate(cfg, mode, cpu_budget, nth)
        rec["cpu_baseline"] = {"value": rate, "unit": "positions/s", "cores": nth, "kind": "oracle",
                               "rounds_per_s": n / el,
                               "sample": f"{n} sequences of the workload in {el:.1f} s, "
                                         f"one oracle call per thread per batch"}
    del sets, outs, graphs, g_iso, g_brk
    torch.cuda.empty_cache()
    return rec


def pool_inputs(w: dict, nsets: int, seed: int = 0):
    """Seeded n-gram steps: ngrams [nsets, B, W, N] and last tokens [nsets, B]."""
    rng = np.random.default_rng(seed)
    B, V, N, W, keys = w["B"], w["V"], w["N"], w["W"], w["keys"]
    ng = rng.integers(0, V, size=(nsets, B, W, N)).astype(np.int32)
    ng[..., 0] = rng.integers(0, keys, size=(nsets, B, W))
    last = rng.integers(0, keys, size=(nsets, B)).astype(np.int32)
    return ng, last


def measure_pool(args, name: str, steps: int, cpu_budget: float, counts: bool):
    """The n-gram pool: one insert of W n-grams per sequence and one lookup
    of G candidates per sequence per step, timed over CUDA-graph replays of
    exactly ``steps`` steps; bit-exact comparison with the oracle's pool over
    the first steps after a reset."""
    import torch
    import speculative_decoding_verification_39_gb300 as svpkg
    w = POOL_WORKLOADS[name]
    B, V, N, cap, G, W = w["B"], w["V"], w["N"], w["cap"], w["G"], w["W"]
    nsets = 64
    ng_h, last_h = pool_inputs(w, nsets)
    dev = torch.device("cuda", torch.cuda.current_device())
    ng = torch.from_numpy(ng_h).to(dev)
    last = torch.from_numpy(last_h).to(dev)
    cand = torch.empty((B, G, N - 1), dtype=torch.int32, device=dev)
    count = torch.empty((B,), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    log(f"[bench] {name}: B={B} W={W} N={N} cap={cap} G={G}")
    rec = {"workload": {"workload": name, "mode": "ngram_pool", "B": B, "V": V, "N": N, "cap": cap, "G": G, "W": W,
                        "l2": "pool and inputs are L2-resident (a few MB); latency-bound"}}
    with torch.cuda.stream(stream):
        pool = svpkg.NgramPool(B, V, N, cap, device=dev)
        if counts:
            # parity: the first nsets steps after a reset, step by step
            ora = __import__("oracle").NgramPool(B, V, N, cap)
            bad = 0
            for i in range(nsets):
                pool.insert(ng[i])
                c, n = pool.lookup(last[i], G, cand=cand, count=count)
                ora.insert(ng_h[i])
                rc, rn = ora.lookup(last_h[i], G)
                bad += int((c.cpu().numpy() != rc).any(axis=(1, 2)).sum() + (n.cpu().numpy() != rn).sum())
            ora.close()
            rec["parity"] = {"steps": nsets, "sequences": B, "lookups": nsets * B, "mismatch": bad,
                             "comparison": "bit-exact candidates and counts against the oracle's pool"}
            log(f"[bench] pool parity: {rec['parity']}")
        pool.reset()
        for i in range(max(3, args.warmup)):
            pool.insert(ng[i % nsets])
            pool.lookup(last[i % nsets], G, cand=cand, count=count)
    stream.synchronize()
    launches_before = svpkg.launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            pool.insert(ng[i % nsets])
            pool.lookup(last[i % nsets], G, cand=cand, count=count)
    captured = svpkg.launch_count() - launches_before
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        t_pre = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - t_pre < 0.5:
                graph.replay()
                stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
    ms_per_step = ms / steps
    peak, peak_kind = measured_peak()
    # bytes a step must touch: per n-gram the key's directory word (read and
    # write), its cap slots (compared) and one slot written; per lookup the
    # directory word, G slots read and G candidates written
    step_bytes = B * W * (8 + cap * (N - 1) * 4 + (N - 1) * 4) + B * (4 + 2 * G * (N - 1) * 4 + 4)
    achieved = step_bytes / (ms_per_step / 1e3) / 1e9
    rec.update({
        "value": B * W * steps / (ms / 1e3),
        "unit": "n-grams inserted/s",
        "lookups_per_s": B * steps / (ms / 1e3),
        "ms_per_step": ms_per_step,
        "steps": steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs", "traffic": pool_traffic(name),
                     "algorithmic_bytes_per_launch": step_bytes, "kernel": "insert_staged_kernel + lookup_kernel",
                     "note": "a few KB per step: the pool is latency-bound (two dependent launches per step), "
                             "not bandwidth-bound",
                     "timing": "CUDA events over one graph of the timed steps"},
        "clocks": clk.summary(),
        "gpu_launches": int(captured),
    })
    if cpu_budget > 0:
        ora = __import__("oracle").NgramPool(B, V, N, cap)
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < cpu_budget:
            ora.insert(ng_h[n % nsets])
            ora.lookup(last_h[n % nsets], G)
            n += 1
        el = time.perf_counter() - t0
        ora.close()
        rec["cpu_baseline"] = {"value": B * W * n / el, "unit": "n-grams inserted/s", "cores": 1, "kind": "oracle",
                               "sample": f"{n} steps in {el:.1f} s on one host thread"}
    del pool, graph
    return rec


def lmhead_inputs(w: dict, dev, seed: int = 0) -> dict:
    """Seeded LM-head inputs on the device: hidden states N(0,1), heads
    N(0,1/D) (bf16), draft tokens drawn from the draft's own logits at T
    (Gumbel-max), uniforms U(0,1)."""
    import torch
    B, K, D, V, T = w["B"], w["K"], w["D"], w["V"], w["T"]
    g = torch.Generator(device=dev).manual_seed(seed)
    ht = torch.randn(B, K + 1, D, device=dev, generator=g).to(torch.bfloat16)
    hd = torch.randn(B, K, D, device=dev, generator=g).to(torch.bfloat16)
    wt = (torch.randn(V, D, device=dev, generator=g) / math.sqrt(D)).to(torch.bfloat16)
    wd = (torch.randn(V, D, device=dev, generator=g) / math.sqrt(D)).to(torch.bfloat16)
    ld = hd.reshape(B * K, D).float() @ wd.float().T
    gum = -torch.log(-torch.log(torch.rand(ld.shape, device=dev, generator=g).clamp_min(1e-30)))
    x = (ld / T + gum).argmax(dim=1).to(torch.int32).reshape(B, K)
    u = torch.rand(B, K + 1, device=dev, generator=g)
    return {"ht": ht, "hd": hd, "wt": wt, "wd": wd, "x": x, "u": u}


def measure_lmhead(args, name: str, steps: int, cpu_budget: float, counts: bool):
    """The verify on LM-head hidden states: one call = the GEMM of both heads
    on the tensor cores (2*(B(K+1)+BK)*V*D flops) and the verify of its fp32
    logits. Timed over a CUDA graph of exactly ``steps`` calls; parity against
    the oracle (fp64 logits) on the first sequences."""
    import torch
    import speculative_decoding_verification_39_gb300 as svpkg
    w = LMHEAD_WORKLOADS[name]
    B, K, D, V, T = w["B"], w["K"], w["D"], w["V"], w["T"]
    dev = torch.device("cuda", torch.cuda.current_device())
    log(f"[bench] {name}: B={B} K={K} D={D} V={V}")
    inp = lmhead_inputs(w, dev)
    stream = torch.cuda.Stream(dev)
    args_t = (inp["ht"], inp["hd"], inp["wt"], inp["wd"], inp["x"], inp["u"], T)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            out = svpkg.verify_sample_lmhead(*args_t)
    stream.synchronize()
    launches_before = svpkg.launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(steps):
            out = svpkg.verify_sample_lmhead(*args_t)
    captured = svpkg.launch_count() - launches_before
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        t_pre = time.perf_counter()
        with torch.cuda.stream(stream):
            while time.perf_counter() - t_pre < 0.5:
                graph.replay()
                stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
    with torch.cuda.stream(stream):
        if svpkg.get_status() != 0:
            raise RuntimeError("device status set by the LM-head verify")
    ms_per_step = ms / steps
    flops = 2.0 * (B * (K + 1) + B * K) * V * D
    tflops = flops / (ms_per_step / 1e3) / 1e12
    peak = measured_bf16_tflops()
    rec = {
        "workload": {"workload": name, "mode": "lmhead_sample", "B": B, "K": K, "D": D, "V": V, "temperature": T,
                     "hidden": "bf16", "l2": "heads (2 x 262 MB) larger than L2"},
        "value": B * (K + 1) / (ms_per_step / 1e3),
        "unit": "positions/s",
        "ms_per_step": ms_per_step,
        "steps": steps,
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak[0], "unit": "TFLOP/s",
                     "frac": tflops / peak[0], "peak_source": peak[1],
                     "traffic": profiled_traffic(name, "lmhead_kernel"),
                     "algorithmic_flops_per_launch": flops, "kernel": "lmhead_kernel",
                     "note": "whole call (the GEMM of both heads and the verify of its fp32 logits) against the "
                             "GEMM's flops: a lower bound on the GEMM kernel's own rate",
                     "timing": "CUDA events over one graph of the timed calls"},
        "clocks": clk.summary(),
        "gpu_launches": int(captured),
    }
    if counts or cpu_budget > 0:
        import oracle
        nb = 4
        host = {k: (v[:nb] if k in ("ht", "hd", "x", "u") else v) for k, v in inp.items()}
        host = {k: (v.view(torch.int16).cpu().numpy().view(np.uint16) if v.dtype == torch.bfloat16 else
                    v.cpu().numpy()) for k, v in host.items()}
        t0 = time.perf_counter()
        ot, oa, om = oracle.verify_sample_lmhead(host["ht"], host["hd"], host["wt"], host["wd"], host["x"], host["u"],
                                                 T)
        el = time.perf_counter() - t0
        gt, ga = out[0][:nb].cpu().numpy(), out[1][:nb].cpu().numpy()
        if counts:
            diff = (gt != ot).any(1) | (ga != oa)
            near = om < 1e-6
            rec["parity"] = {"sequences": nb, "mismatch": int(diff.sum()),
                             "mismatch_away_from_near_tie": int((diff & ~near).sum()), "near_ties": int(near.sum()),
                             "comparison": "tokens and accept lengths against the oracle's verify on fp64 logits "
                                           "of the same bf16 hidden states and heads (differences only at "
                                           "near-ties: the GPU accumulates in fp32)"}
        if cpu_budget > 0:
            rec["cpu_baseline"] = {"value": nb * (K + 1) / el, "unit": "positions/s", "cores": 1, "kind": "oracle",
                                   "sample": f"{nb} sequences (fp64 GEMV of both heads, then the verify) in {el:.1f} s"}
    del graph
    return rec


def measured_bf16_tflops():
    """(bf16 TFLOP/s, source): the burst figure of MEASURED_PEAKS.json, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            v = float(json.load(fh)["bf16_tflops"])
        return v, "measured bf16_tflops (burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback bf16"


def run_calls(args, name: str):
    """``--calls N``: N plain calls of one workload on the current stream, then
    exit (for profilers: no graphs, no timing, no oracle)."""
    import torch
    import speculative_decoding_verification_39_gb300 as svpkg
    torch.cuda.set_device(0)
    svpkg.build()
    svpkg.set_greedy_path(args.greedy_path)
    svpkg.set_sample_path(args.sample_path)
    dev = torch.device("cuda", 0)
    n = args.calls
    if name in POOL_WORKLOADS:
        w = POOL_WORKLOADS[name]
        ng, last = pool_inputs(w, n)
        pool = svpkg.NgramPool(w["B"], w["V"], w["N"], w["cap"], device=dev)
        ng, last = torch.from_numpy(ng).to(dev), torch.from_numpy(last).to(dev)
        for i in range(n):
            pool.insert(ng[i])
            pool.lookup(last[i], w["G"])
    elif name in LMHEAD_WORKLOADS:
        w = LMHEAD_WORKLOADS[name]
        inp = lmhead_inputs(w, dev)
        for _ in range(n):
            svpkg.verify_sample_lmhead(inp["ht"], inp["hd"], inp["wt"], inp["wd"], inp["x"], inp["u"], w["T"])
    else:
        cfg, mode = workload(name, args.batch)[:2]
        host = host_inputs(cfg, mode)
        keys = {"greedy": ("logits", "cand"), "lookahead": ("logits", "cand", "uniforms"),
                "multidraft": ("target", "draft", "draft_tokens", "uniforms"),
                "sample": ("target", "draft", "draft_tokens", "uniforms")}[mode]
        t = [to_torch(host[k], torch).to(dev) for k in keys]
        for _ in range(n):
            if mode == "greedy":
                svpkg.verify_greedy(*t)
            elif mode == "lookahead":
                svpkg.verify_lookahead_sample(*t, cfg.temperature)
            elif mode == "multidraft":
                svpkg.verify_multidraft_sample(*t, cfg.temperature)
            else:
                svpkg.verify_sample(*t, cfg.temperature, cfg.top_p)
    torch.cuda.synchronize()
    if svpkg.get_status() != 0:
        raise RuntimeError("device status set")
    log(f"[bench] {n} calls of {name}; refined draws so far: {svpkg.refined_draws()}")


def run_gpu(args, names: list, rank: int, world: int):
    import torch
    import speculative_decoding_verification_39_gb300 as svpkg

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(torch.device("cuda", local))
    svpkg.build()
    svpkg.set_greedy_path(args.greedy_path)
    svpkg.set_sample_path(args.sample_path)
    head = names[0]
    if head in EXTRA_WORKLOADS:
        raise SystemExit(f"{head} is not a verify call of logits: name it after one (its record is a per_config one)")
    rec = measure(args, head, rank, world, args.steps, 0.0 if args.no_cpu_baseline else args.cpu_budget,
                  counts=not args.no_counts)
    cfg, mode = workload(head, args.batch)[:2]
    line = {
        "metric": "verified positions/sec and achieved HBM GB/s (% of GB300 peak) per verify call",
        "value": rec["value"],
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded Philox inputs of the workload's shapes)",
        "config": rec["workload"],
    }
    for k in ("rounds_per_s", "isolated_us", "isolated_note", "roofline", "clocks", "e2e", "gpu_launches",
              "refined_draws_per_call", "refined_note", "parity", "cpu_baseline"):
        if k in rec:
            line[k] = rec[k]
    if "cpu_baseline" in line and not args.no_cpu_baseline and rank == 0 and world == 1:
        rate1, n1, el1 = oracle_cpu_rate(cfg, mode, args.cpu_budget / 2, 1)
        line["cpu_baseline"]["single_thread"] = {"value": rate1, "unit": "positions/s", "cores": 1,
                                                 "rounds_per_s": n1 / el1, "sample": f"{n1} sequences in {el1:.1f} s"}
    if len(names) > 1 and world == 1:
        per = {}
        for n in names[1:]:
            if n in POOL_WORKLOADS:
                r = measure_pool(args, n, max(args.steps, 100), 0.0 if args.no_cpu_baseline else 2.0,
                                 counts=not args.no_counts)
            elif n in LMHEAD_WORKLOADS:
                r = measure_lmhead(args, n, max(args.steps, 100), 0.0 if args.no_cpu_baseline else 2.0,
                                   counts=not args.no_counts)
            else:
                r = measure(args, n, rank, world, max(args.steps, 100), 0.0 if args.no_cpu_baseline else 2.0,
                            counts=not args.no_counts)
            per[n] = r
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    return line


# ---------------------------------------------------------- reference arm

def run_reference(args, name: str):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    cfg, mode, positions, logit_bytes, _, _ = workload(name, args.batch)
    nth = os.cpu_count() or 1
    per_step = max(5.0, 60.0 / max(1, args.steps + args.warmup))
    rates, rounds = [], []
    for i in range(args.warmup + args.steps):
        rate, n, el = oracle_cpu_rate(cfg, mode, min(per_step, 20.0), nth)
        if i >= args.warmup:
            rates.append(rate)
            rounds.append(n / el)
    value = float(np.mean(rates))
    line = {
        "impl": "reference",
        "metric": "verified positions/sec and achieved HBM GB/s (% of GB300 peak) per verify call",
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": positions / value * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded Philox inputs of the workload's shapes)",
        "config": config_json(cfg, mode, 1),
        "rounds_per_s": float(np.mean(rounds)),
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": nth, "kind": "oracle",
                         "sample": f"per step: a bounded sample of the workload's sequences, about "
                                   f"{min(per_step, 20.0):.0f} s of CPU work"},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def all_names() -> list:
    return (list(sg.CONFIGS) + list(sg.LOOKAHEAD_CONFIGS) + list(sg.MULTIDRAFT_CONFIGS) + list(POOL_WORKLOADS) +
            list(LMHEAD_WORKLOADS))


def config_names(spec) -> list:
    """None: the headline workload, then every other one (their per_config
    records); 'all': the same; otherwise one workload name or several
    separated by commas (the first is the line's own)."""
    if spec is None or spec == "all":
        return [DEFAULT_CONFIG] + [n for n in all_names() if n != DEFAULT_CONFIG]
    names = [n.strip() for n in spec.split(",") if n.strip()]
    for n in names:
        if n not in EXTRA_WORKLOADS:
            find_config(n)  # KeyError for an unknown name, before any work
    return names


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=None,
                    help="workload name, several joined by commas (the first is the line's own, the rest its "
                         "per_config records), or 'all' (the default: the headline workload, then every other)")
    ap.add_argument("--no-counts", action="store_true", help="skip the GPU/oracle mismatch counts")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of CPU oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (--batch 1: per-call latency of one sequence)")
    ap.add_argument("--greedy-path", type=int, default=0, choices=[0, 1],
                    help="greedy verify kernels: 0 row argmax + match kernels, 1 the streaming kernel")
    ap.add_argument("--sample-path", type=int, default=0, choices=[0, 1, 2],
                    help="sampling verify kernels: 0 by the library's size rule, 1 the streaming kernel, 2 the row "
                         "pass + cluster decide kernel wherever they fit")
    ap.add_argument("--l2-resident", action="store_true",
                    help="replay one input set, so that inputs that fit stay in L2 (reported as such; not an "
                         "HBM figure)")
    ap.add_argument("--calls", type=int, default=0,
                    help="run this many plain calls of the first named workload and exit (for profilers)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    names = config_names(args.config)
    if args.calls > 0:
        run_calls(args, names[0])
        return
    if args.impl == "reference":
        run_reference(args, names[0])
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world != args.gpus:
        log(f"[bench] --gpus {args.gpus} but WORLD_SIZE {world}; using WORLD_SIZE")
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    try:
        run_gpu(args, names, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
