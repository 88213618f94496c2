"""Seeded synthetic inputs for the speculative-decoding verify step.

This module only makes inputs. The CPU oracle's tests and the GPU benchmark
both read its arrays, so the two sides see identical bytes; it holds none of
the verify step's arithmetic. Random numbers come from Philox4x32-10
(counter-based), keyed by (seed, stream) with the flat element index as the
counter, so a batch generated in shards (``seq_offset``) equals the same batch
generated whole.

Storage convention for logits: ``dtype`` 0 is fp32 (numpy float32), ``dtype``
1 is bf16 stored as its raw 16-bit pattern (numpy uint16).

The five workloads are those the verify step is measured on; see ``CONFIGS``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specgen.c")
_SO = os.path.join(_HERE, "libspecgen.so")

F32 = 0
BF16 = 1

STREAM_UNIFORM = 5


def build(force: bool = False) -> str:
    """Compile ``libspecgen.so`` next to its source (plain C, no GPU)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared",
             "-pthread", _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, _SO)
    return _SO


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        i64, i32, u64, f32, f64, vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_void_p)
        lib.sg_philox4x32_10.argtypes = [vp, vp, vp]
        lib.sg_philox4x32_10.restype = None
        lib.sg_gen_logits.argtypes = [vp, vp, ctypes.c_int, i64, i32, i64, f64, f64, i32, f64, u64, i64, i32]
        lib.sg_gen_logits.restype = ctypes.c_int
        lib.sg_draft_tokens.argtypes = [vp, ctypes.c_int, i64, i32, i64, f32, f32, u64, i64, vp, i32]
        lib.sg_draft_tokens.restype = ctypes.c_int
        lib.sg_uniforms.argtypes = [i64, i32, u64, i64, vp]
        lib.sg_uniforms.restype = ctypes.c_int
        lib.sg_gen_greedy.argtypes = [vp, vp, ctypes.c_int, i64, i32, i32, i64, f64, f64, u64, i64, i32]
        lib.sg_gen_greedy.restype = ctypes.c_int
        lib.sg_uniform_doubles.argtypes = [u64, ctypes.c_uint32, u64, i64, vp]
        lib.sg_uniform_doubles.restype = ctypes.c_int
        _lib_handle = lib
    return _lib_handle


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def np_dtype(dtype: int):
    return np.uint16 if dtype == BF16 else np.float32


def philox4x32_10(ctr, key) -> tuple:
    """One Philox4x32-10 block: 4 x uint32 counter, 2 x uint32 key -> 4 x uint32."""
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _lib().sg_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return tuple(int(x) for x in out)


def to_float(a: np.ndarray, dtype: int) -> np.ndarray:
    """Stored logits -> float64 values (bf16 bit patterns are widened exactly)."""
    if dtype == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def from_float(x: np.ndarray, dtype: int) -> np.ndarray:
    """float values -> stored logits, rounding to nearest even for bf16."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F32:
        return f
    u = f.view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def uniforms(B: int, K: int, seed: int = 0, seq_offset: int = 0) -> np.ndarray:
    """uniforms[B, K+1] fp32 in [0, 1): K accept tests and one sample draw per sequence."""
    out = np.empty((B, K + 1), dtype=np.float32)
    assert _lib().sg_uniforms(B, K, seed, seq_offset, _ptr(out)) == 0
    return out


def uniform_doubles(n: int, seed: int = 0, stream: int = 99, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    assert _lib().sg_uniform_doubles(seed, stream, first, n, _ptr(out)) == 0
    return out


def draft_tokens(draft: np.ndarray, dtype: int, temperature: float, top_p: float = 1.0, seed: int = 0,
                 seq_offset: int = 0, nthreads: int = 0) -> np.ndarray:
    """One draw per draft row of ``draft[B, K, V]`` from softmax(l/T) (top-p filtered).

    This stands in for the draft model's own sampler; T == 0 takes the argmax.
    """
    draft = np.ascontiguousarray(draft)
    B, K, V = draft.shape
    out = np.empty((B, K), dtype=np.int32)
    rc = _lib().sg_draft_tokens(_ptr(draft), dtype, B, K, V, float(temperature), float(top_p), seed, seq_offset,
                                _ptr(out), nthreads)
    assert rc == 0
    return out


@dataclass(frozen=True)
class SampleConfig:
    """A sampling-mode verify workload: target [B,K+1,V], draft [B,K,V]."""
    name: str
    B: int
    K: int
    V: int
    dtype: int
    temperature: float
    top_p: float
    target_sigma: float
    peak_height: float
    n_peaks: int
    draft_sigma: float
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.B * (2 * self.K + 1)

    @property
    def logit_bytes(self) -> int:
        return self.rows * self.V * (2 if self.dtype == BF16 else 4)

    def with_(self, **kw) -> "SampleConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class GreedyConfig:
    """A greedy (Lookahead) verify workload: logits [B,G,N,V], cand [B,G,N-1]."""
    name: str
    B: int
    G: int
    N: int
    V: int
    dtype: int
    sigma: float
    match_prob: float
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.B * self.G * self.N

    @property
    def logit_bytes(self) -> int:
        return self.rows * self.V * (2 if self.dtype == BF16 else 4)

    def with_(self, **kw) -> "GreedyConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class LookaheadSampleConfig:
    """A Lookahead sampling-mode verify workload: logits [B,G,N,V] and cand
    [B,G,N-1] made as for the greedy workload (candidates are produced
    greedily), uniforms [B,(N-1)*G+1], temperature > 0."""
    name: str
    B: int
    G: int
    N: int
    V: int
    dtype: int
    sigma: float
    match_prob: float
    temperature: float
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.B * self.G * self.N

    @property
    def logit_bytes(self) -> int:
        return self.rows * self.V * (2 if self.dtype == BF16 else 4)

    def with_(self, **kw) -> "LookaheadSampleConfig":
        return replace(self, **kw)


# The five measured workloads. The first one's "1000 rounds of B=1" are 1000
# independent sequences, verified as one batch of 1000.
CONFIGS = {
    "cfg1_v1000_f32": SampleConfig("cfg1_v1000_f32", B=1000, K=4, V=1000, dtype=F32, temperature=1.0, top_p=1.0,
                                   target_sigma=3.0, peak_height=6.0, n_peaks=5, draft_sigma=1.0),
    "cfg2_v32000_bf16": SampleConfig("cfg2_v32000_bf16", B=64, K=5, V=32000, dtype=BF16, temperature=1.0,
                                     top_p=1.0, target_sigma=3.0, peak_height=6.0, n_peaks=5, draft_sigma=0.7),
    "cfg3_v128256_bf16": SampleConfig("cfg3_v128256_bf16", B=256, K=8, V=128256, dtype=BF16, temperature=0.8,
                                      top_p=1.0, target_sigma=3.0, peak_height=5.0, n_peaks=8, draft_sigma=1.2),
    "cfg4_greedy_v32000_bf16": GreedyConfig("cfg4_greedy_v32000_bf16", B=32, G=7, N=5, V=32000, dtype=BF16,
                                            sigma=3.0, match_prob=0.5),
    "cfg5_topp_v151936_bf16": SampleConfig("cfg5_topp_v151936_bf16", B=128, K=6, V=151936, dtype=BF16,
                                           temperature=0.7, top_p=0.9, target_sigma=2.5, peak_height=5.0,
                                           n_peaks=10, draft_sigma=0.8),
}


@dataclass(frozen=True)
class MultiDraftConfig:
    """A multi-draft sampling verify workload: target [B,G,N,V], draft
    [B,G,N-1,V], draft_tokens [B,G,N-1] drawn from the draft rows, uniforms
    [B,(N-1)*G+1]. Each (sequence, draft) pair is made like one sampling-mode
    sequence with K = N-1: target rows sigma*N(0,1) with n_peaks raised by
    peak_height, draft rows = target + draft_sigma*N(0,1)."""
    name: str
    B: int
    G: int
    N: int
    V: int
    dtype: int
    temperature: float
    target_sigma: float
    peak_height: float
    n_peaks: int
    draft_sigma: float
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.B * self.G * (2 * self.N - 1)

    @property
    def logit_bytes(self) -> int:
        return self.rows * self.V * (2 if self.dtype == BF16 else 4)

    def with_(self, **kw) -> "MultiDraftConfig":
        return replace(self, **kw)


MULTIDRAFT_CONFIGS = {
    "md_sample_v32000_bf16": MultiDraftConfig("md_sample_v32000_bf16", B=32, G=7, N=5, V=32000, dtype=BF16,
                                              temperature=1.0, target_sigma=3.0, peak_height=6.0, n_peaks=5,
                                              draft_sigma=0.7),
}


# The Lookahead sampling-mode verify on the greedy workload's shape, at the
# temperature the Lookahead page's sampling experiments use (1.0).
LOOKAHEAD_CONFIGS = {
    "la_sample_v32000_bf16": LookaheadSampleConfig("la_sample_v32000_bf16", B=32, G=7, N=5, V=32000, dtype=BF16,
                                                   sigma=3.0, match_prob=0.5, temperature=1.0),
}


def sample_inputs(cfg: SampleConfig, seq_offset: int = 0, B: int | None = None, nthreads: int = 0,
                  out: dict | None = None) -> dict:
    """Generate target, draft, draft_tokens and uniforms for ``cfg``.

    ``B`` overrides the batch size (a shard of ``cfg.B`` sequences starting at
    global sequence ``seq_offset``). ``out`` may supply preallocated arrays
    (e.g. views of pinned host memory) under the same keys.
    """
    B = cfg.B if B is None else B
    dt = np_dtype(cfg.dtype)
    out = {} if out is None else out
    target = out.setdefault("target", np.empty((B, cfg.K + 1, cfg.V), dtype=dt))
    draft = out.setdefault("draft", np.empty((B, cfg.K, cfg.V), dtype=dt))
    rc = _lib().sg_gen_logits(_ptr(target), _ptr(draft), cfg.dtype, B, cfg.K, cfg.V, cfg.target_sigma,
                              cfg.peak_height, cfg.n_peaks, cfg.draft_sigma, cfg.seed, seq_offset, nthreads)
    assert rc == 0
    toks = out.setdefault("draft_tokens", np.empty((B, cfg.K), dtype=np.int32))
    rc = _lib().sg_draft_tokens(_ptr(draft), cfg.dtype, B, cfg.K, cfg.V, float(cfg.temperature), float(cfg.top_p),
                                cfg.seed, seq_offset, _ptr(toks), nthreads)
    assert rc == 0
    u = out.setdefault("uniforms", np.empty((B, cfg.K + 1), dtype=np.float32))
    assert _lib().sg_uniforms(B, cfg.K, cfg.seed, seq_offset, _ptr(u)) == 0
    return out


def greedy_inputs(cfg: GreedyConfig, seq_offset: int = 0, B: int | None = None, nthreads: int = 0,
                  out: dict | None = None) -> dict:
    """Generate logits [B,G,N,V] and cand [B,G,N-1] for ``cfg``."""
    B = cfg.B if B is None else B
    out = {} if out is None else out
    logits = out.setdefault("logits", np.empty((B, cfg.G, cfg.N, cfg.V), dtype=np_dtype(cfg.dtype)))
    cand = out.setdefault("cand", np.empty((B, cfg.G, cfg.N - 1), dtype=np.int32))
    rc = _lib().sg_gen_greedy(_ptr(logits), _ptr(cand), cfg.dtype, B, cfg.G, cfg.N, cfg.V, cfg.sigma,
                              cfg.match_prob, cfg.seed, seq_offset, nthreads)
    assert rc == 0
    return out


def lookahead_sample_inputs(cfg: LookaheadSampleConfig, seq_offset: int = 0, B: int | None = None,
                            nthreads: int = 0, out: dict | None = None) -> dict:
    """Generate logits [B,G,N,V], cand [B,G,N-1] and uniforms [B,(N-1)*G+1] for ``cfg``."""
    B = cfg.B if B is None else B
    out = greedy_inputs(GreedyConfig(cfg.name, B=B, G=cfg.G, N=cfg.N, V=cfg.V, dtype=cfg.dtype, sigma=cfg.sigma,
                                     match_prob=cfg.match_prob, seed=cfg.seed),
                        seq_offset=seq_offset, B=B, nthreads=nthreads, out=out)
    u = out.setdefault("uniforms", np.empty((B, (cfg.N - 1) * cfg.G + 1), dtype=np.float32))
    assert _lib().sg_uniforms(B, (cfg.N - 1) * cfg.G, cfg.seed, seq_offset, _ptr(u)) == 0
    return out


def multidraft_inputs(cfg: MultiDraftConfig, seq_offset: int = 0, B: int | None = None, nthreads: int = 0) -> dict:
    """Generate target, draft, draft_tokens and uniforms for ``cfg``; shards
    (``seq_offset``) equal the same batch generated whole."""
    B = cfg.B if B is None else B
    G, N = cfg.G, cfg.N
    dt = np_dtype(cfg.dtype)
    target = np.empty((B * G, N, cfg.V), dtype=dt)
    draft = np.empty((B * G, N - 1, cfg.V), dtype=dt)
    rc = _lib().sg_gen_logits(_ptr(target), _ptr(draft), cfg.dtype, B * G, N - 1, cfg.V, cfg.target_sigma,
                              cfg.peak_height, cfg.n_peaks, cfg.draft_sigma, cfg.seed, seq_offset * G, nthreads)
    assert rc == 0
    toks = np.empty((B * G, N - 1), dtype=np.int32)
    rc = _lib().sg_draft_tokens(_ptr(draft), cfg.dtype, B * G, N - 1, cfg.V, float(cfg.temperature), 1.0, cfg.seed,
                                seq_offset * G, _ptr(toks), nthreads)
    assert rc == 0
    u = np.empty((B, (N - 1) * G + 1), dtype=np.float32)
    assert _lib().sg_uniforms(B, (N - 1) * G, cfg.seed, seq_offset, _ptr(u)) == 0
    return {"target": target.reshape(B, G, N, cfg.V), "draft": draft.reshape(B, G, N - 1, cfg.V),
            "draft_tokens": toks.reshape(B, G, N - 1), "uniforms": u}
