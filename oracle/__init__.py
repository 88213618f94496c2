"""Python access to the CPU oracle of the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY. The oracle (``oracle.c``, plain fp64 C) is what the
GPU library is checked against. Only the test suite, the package's smoke
check and the benchmark's CPU-baseline leg may import this module. The GPU
library shares no code with it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_SO = os.path.join(_HERE, "liboracle.so")


def compile_oracle(src: str, out: str, extra_flags=()) -> str:
    """Compile an oracle source file into a shared library (plain C, fp64)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", *extra_flags, "-I", _HERE,
                    src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        compile_oracle(_SRC, _SO)
    return _SO


def _bind(lib):
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    lib.oracle_verify_sample.argtypes = [vp, vp, ctypes.c_int, vp, vp, i64, i32, i64, f32, f32, vp, vp, vp]
    lib.oracle_verify_sample.restype = ctypes.c_int
    lib.oracle_row_stats.argtypes = [vp, ctypes.c_int, i64, i64, f32, f32, vp]
    lib.oracle_row_stats.restype = ctypes.c_int
    lib.oracle_verify_greedy.argtypes = [vp, ctypes.c_int, vp, i64, i32, i32, i64, vp, vp, vp]
    lib.oracle_verify_greedy.restype = ctypes.c_int
    lib.oracle_verify_lookahead_sample.argtypes = [vp, ctypes.c_int, vp, vp, i64, i32, i32, i64, f32, vp, vp, vp,
                                                   vp]
    lib.oracle_verify_lookahead_sample.restype = ctypes.c_int
    lib.oracle_verify_multidraft_sample.argtypes = [vp, vp, ctypes.c_int, vp, vp, i64, i32, i32, i64, f32, vp, vp,
                                                    vp, vp]
    lib.oracle_verify_multidraft_sample.restype = ctypes.c_int
    lib.oracle_verify_sample_lmhead.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, vp, i64, i32, i64, i64, f32, f32,
                                                vp, vp, vp]
    lib.oracle_verify_sample_lmhead.restype = ctypes.c_int
    lib.oracle_ngram_pool_create.argtypes = [i64, i64, i32, i32]
    lib.oracle_ngram_pool_create.restype = vp
    lib.oracle_ngram_pool_destroy.argtypes = [vp]
    lib.oracle_ngram_pool_destroy.restype = None
    lib.oracle_ngram_pool_insert.argtypes = [vp, vp, i32]
    lib.oracle_ngram_pool_insert.restype = ctypes.c_int
    lib.oracle_ngram_pool_lookup.argtypes = [vp, vp, i32, vp, vp]
    lib.oracle_ngram_pool_lookup.restype = ctypes.c_int
    lib.oracle_inverse_cdf.argtypes = [vp, i64, ctypes.c_double, vp]
    lib.oracle_inverse_cdf.restype = ctypes.c_int
    lib.oracle_residual_draw.argtypes = [vp, vp, i64, ctypes.c_double, vp]
    lib.oracle_residual_draw.restype = ctypes.c_int
    return lib


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _bind(ctypes.CDLL(build()))
    return _lib_handle


def load_library(path: str):
    """Bind an alternative build of the oracle (used by the mutation tests)."""
    return _bind(ctypes.CDLL(path))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float32:
        return 0
    raise TypeError(f"logits must be float32 or bf16 bit patterns (uint16), got {a.dtype}")


def verify_sample(target, draft, draft_tokens, uniforms, temperature: float, top_p: float = 1.0, lib=None):
    """Sampling-mode verify of a batch. Returns (tokens[B,K+1], accept_len[B], margin[B])."""
    lib = lib or _lib()
    target = np.ascontiguousarray(target)
    B, K1, V = target.shape
    K = K1 - 1
    draft = np.ascontiguousarray(draft) if draft is not None else np.zeros((B, K, V), dtype=target.dtype)
    assert draft.shape == (B, K, V) and draft.dtype == target.dtype
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    u = np.ascontiguousarray(uniforms, dtype=np.float32) if uniforms is not None else np.zeros((B, K1), np.float32)
    out = np.empty((B, K1), dtype=np.int32)
    acc = np.empty(B, dtype=np.int32)
    margin = np.empty(B, dtype=np.float64)
    rc = lib.oracle_verify_sample(_p(target), _p(draft), _dtype_code(target), _p(toks), _p(u), B, K, V,
                                  float(temperature), float(top_p), _p(out), _p(acc), _p(margin))
    if rc != 0:
        raise ValueError("oracle_verify_sample: argument error")
    return out, acc, margin


def row_stats(rows, temperature: float, top_p: float = 1.0, lib=None):
    """Per-row {m, lse, P_S, tau} of rows[..., V] (float64 [..., 4])."""
    lib = lib or _lib()
    rows = np.ascontiguousarray(rows)
    V = rows.shape[-1]
    n = rows.size // V
    out = np.empty((n, 4), dtype=np.float64)
    rc = lib.oracle_row_stats(_p(rows), _dtype_code(rows), n, V, float(temperature), float(top_p), _p(out))
    if rc != 0:
        raise ValueError("oracle_row_stats: argument error")
    return out.reshape(rows.shape[:-1] + (4,))


def verify_greedy(logits, cand, lib=None):
    """Greedy verify. Returns (tokens[B,N], accept_len[B], best[B])."""
    lib = lib or _lib()
    logits = np.ascontiguousarray(logits)
    B, G, N, V = logits.shape
    cand = np.ascontiguousarray(cand, dtype=np.int32)
    assert cand.shape == (B, G, N - 1)
    out = np.empty((B, N), dtype=np.int32)
    acc = np.empty(B, dtype=np.int32)
    best = np.empty(B, dtype=np.int32)
    rc = lib.oracle_verify_greedy(_p(logits), _dtype_code(logits), _p(cand), B, G, N, V, _p(out), _p(acc), _p(best))
    if rc != 0:
        raise ValueError("oracle_verify_greedy: argument error")
    return out, acc, best


def verify_lookahead_sample(logits, cand, uniforms, temperature: float, lib=None):
    """Lookahead sampling-mode verify of greedily produced candidates.
    Returns (tokens[B,N], accept_len[B], best[B], margin[B])."""
    lib = lib or _lib()
    logits = np.ascontiguousarray(logits)
    B, G, N, V = logits.shape
    cand = np.ascontiguousarray(cand, dtype=np.int32)
    assert cand.shape == (B, G, N - 1)
    u = np.ascontiguousarray(uniforms, dtype=np.float32)
    assert u.shape == (B, (N - 1) * G + 1)
    out = np.empty((B, N), dtype=np.int32)
    acc = np.empty(B, dtype=np.int32)
    best = np.empty(B, dtype=np.int32)
    margin = np.empty(B, dtype=np.float64)
    rc = lib.oracle_verify_lookahead_sample(_p(logits), _dtype_code(logits), _p(cand), _p(u), B, G, N, V,
                                            float(temperature), _p(out), _p(acc), _p(best), _p(margin))
    if rc != 0:
        raise ValueError("oracle_verify_lookahead_sample: argument error")
    return out, acc, best, margin


def verify_multidraft_sample(target, draft, draft_tokens, uniforms, temperature: float, lib=None):
    """Multi-draft sampling verify: target [B,G,N,V], draft [B,G,N-1,V],
    draft_tokens [B,G,N-1], uniforms [B,(N-1)*G+1].
    Returns (tokens[B,N], accept_len[B], best[B], margin[B])."""
    lib = lib or _lib()
    target = np.ascontiguousarray(target)
    B, G, N, V = target.shape
    draft = np.ascontiguousarray(draft)
    assert draft.shape == (B, G, N - 1, V) and draft.dtype == target.dtype
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    assert toks.shape == (B, G, N - 1)
    u = np.ascontiguousarray(uniforms, dtype=np.float32)
    assert u.shape == (B, (N - 1) * G + 1)
    out = np.empty((B, N), dtype=np.int32)
    acc = np.empty(B, dtype=np.int32)
    best = np.empty(B, dtype=np.int32)
    margin = np.empty(B, dtype=np.float64)
    rc = lib.oracle_verify_multidraft_sample(_p(target), _p(draft), _dtype_code(target), _p(toks), _p(u), B, G, N,
                                             V, float(temperature), _p(out), _p(acc), _p(best), _p(margin))
    if rc != 0:
        raise ValueError("oracle_verify_multidraft_sample: argument error")
    return out, acc, best, margin


def verify_sample_lmhead(h_target, h_draft, w_target, w_draft, draft_tokens, uniforms, temperature: float,
                         top_p: float = 1.0, lib=None):
    """Sampling verify on logits h · W^T computed in fp64 from hidden states
    h_target [B,K+1,D], h_draft [B,K,D] and LM heads w_target, w_draft [V,D].
    Returns (tokens[B,K+1], accept_len[B], margin[B])."""
    lib = lib or _lib()
    ht, hd = np.ascontiguousarray(h_target), np.ascontiguousarray(h_draft)
    wt, wd = np.ascontiguousarray(w_target), np.ascontiguousarray(w_draft)
    B, K1, D = ht.shape
    K = K1 - 1
    V = wt.shape[0]
    assert hd.shape == (B, K, D) and wt.shape == (V, D) and wd.shape == (V, D)
    assert ht.dtype == hd.dtype == wt.dtype == wd.dtype
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    u = np.ascontiguousarray(uniforms, dtype=np.float32)
    out = np.empty((B, K1), dtype=np.int32)
    acc = np.empty(B, dtype=np.int32)
    margin = np.empty(B, dtype=np.float64)
    rc = lib.oracle_verify_sample_lmhead(_p(ht), _p(hd), _p(wt), _p(wd), _dtype_code(ht), _p(toks), _p(u), B, K, D, V,
                                         float(temperature), float(top_p), _p(out), _p(acc), _p(margin))
    if rc != 0:
        raise ValueError("oracle_verify_sample_lmhead: argument error")
    return out, acc, margin


def inverse_cdf(w, u: float, lib=None) -> int:
    """The oracle's inverse-CDF draw from unnormalised weights (test-only entry)."""
    lib = lib or _lib()
    w = np.ascontiguousarray(w, dtype=np.float64)
    out = np.zeros(1, dtype=np.int64)
    if lib.oracle_inverse_cdf(_p(w), w.size, float(u), _p(out)) != 0:
        raise ValueError("oracle_inverse_cdf: argument error")
    return int(out[0])


def residual_draw(p, q, u: float, lib=None) -> int:
    """The oracle's draw after a rejection: max(0, p - q), or p if that is all zero."""
    lib = lib or _lib()
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    assert p.shape == q.shape
    out = np.zeros(1, dtype=np.int64)
    if lib.oracle_residual_draw(_p(p), _p(q), p.size, float(u), _p(out)) != 0:
        raise ValueError("oracle_residual_draw: argument error")
    return int(out[0])


class NgramPool:
    """The oracle's n-gram pool (one per sequence, keyed by first token)."""

    def __init__(self, B: int, V: int, N: int, cap: int, lib=None):
        self.lib = lib or _lib()
        self.B, self.V, self.N, self.cap = B, V, N, cap
        self.h = self.lib.oracle_ngram_pool_create(B, V, N, cap)
        if not self.h:
            raise ValueError("oracle_ngram_pool_create: argument error")

    def insert(self, ngrams):
        g = np.ascontiguousarray(ngrams, dtype=np.int32)
        assert g.ndim == 3 and g.shape[0] == self.B and g.shape[2] == self.N
        if self.lib.oracle_ngram_pool_insert(self.h, _p(g), g.shape[1]) != 0:
            raise ValueError("oracle_ngram_pool_insert: argument error")

    def lookup(self, last, G: int):
        last = np.ascontiguousarray(last, dtype=np.int32)
        cand = np.empty((self.B, G, self.N - 1), dtype=np.int32)
        count = np.empty(self.B, dtype=np.int32)
        if self.lib.oracle_ngram_pool_lookup(self.h, _p(last), G, _p(cand), _p(count)) != 0:
            raise ValueError("oracle_ngram_pool_lookup: argument error")
        return cand, count

    def close(self):
        if self.h:
            self.lib.oracle_ngram_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()
