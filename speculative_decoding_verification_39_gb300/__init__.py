"""libspecverify — the speculative-decoding verify step on GB300 (sm_103a).

This module is a thin binding over the C ABI in ``include/specverify.h``: it
checks and marshals torch tensors (device memory, the current stream) into the
library's entry points, which run every step of the verify path in the CUDA
kernels of ``csrc/``. There is no CPU fallback: if ``libspecverify.so`` is
missing or cannot be loaded, every call raises.

Entry points (same names as the C ABI):
  verify_sample(target, draft, draft_tokens, uniforms, temperature, top_p)
  verify_greedy(logits, cand)
  verify_lookahead_sample(logits, cand, uniforms, temperature)
  verify_multidraft_sample(target, draft, draft_tokens, uniforms, temperature)
  get_status()
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(os.path.dirname(_HERE), "include")
_SO = os.path.join(_HERE, "libspecverify.so")
_SOURCES = ["sv_kernels.cu", "sv_api.cu", "sv_noalloc.cu", "sv_lookahead.cu", "sv_multidraft.cu",
            "sv_greedy_rows.cu", "sv_rows.cu", "sv_decide.cu", "sv_ngram.cu", "sv_refine.cu", "sv_lmhead.cu"]
_DEPS = _SOURCES + ["sv_kernels.h", "sv_device.cuh", "sv_lookahead.h", "sv_multidraft.h", "sv_rowstat.cuh",
                    "sv_greedy_rows.h", "sv_v2.h", "sv_df.cuh", "sv_sample_impl.h",
                    "sv_refine.h", "sv_lmhead.h"]

SV_F32, SV_BF16 = 0, 1
STATUS = {0: "SV_OK", -1: "SV_ERR_ARG", -2: "SV_ERR_DTYPE", -3: "SV_ERR_CUDA", -4: "SV_ERR_INPUT",
          -5: "SV_ERR_TIMEOUT", -6: "SV_ERR_NOMEM", -7: "SV_ERR_SCRATCH_LIMIT"}

NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC"]


class SpecVerifyError(RuntimeError):
    def __init__(self, rc: int, what: str):
        super().__init__(f"{what}: {STATUS.get(rc, rc)}")
        self.rc = rc


def _stale() -> bool:
    if not os.path.exists(_SO):
        return True
    t = os.path.getmtime(_SO)
    deps = [os.path.join(_CSRC, f) for f in _DEPS] + [os.path.join(_INCLUDE, "specverify.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libspecverify.so`` in-tree for sm_103a (nvcc; no GPU needed)."""
    if not force and not _stale():
        return _SO
    objs = []

    def cc(src):
        obj = os.path.join(_CSRC, os.path.splitext(src)[0] + f".{os.getpid()}.o")
        cmd = ["nvcc", *NVCC_FLAGS, "-c", os.path.join(_CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(len(_SOURCES)) as ex:
        objs = list(ex.map(cc, _SOURCES))
    tmp = _SO + f".tmp{os.getpid()}"
    try:
        subprocess.run(["nvcc", "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp],
                       check=True, capture_output=True, text=True)
        os.replace(tmp, _SO)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return _SO


_lib_handle = None


def lib():
    """The loaded ``libspecverify.so``; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_SO):
            raise RuntimeError(f"libspecverify.so is not built ({_SO}); run __graft_entry__.build()")
        h = ctypes.CDLL(_SO)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        h.sv_verify_sample.argtypes = [vp, vp, vp, vp, i64, i32, i64, i32, f32, f32, vp, vp, vp, vp]
        h.sv_verify_sample.restype = ctypes.c_int
        h.sv_verify_greedy.argtypes = [vp, vp, i64, i32, i32, i64, i32, vp, vp, vp, vp]
        h.sv_verify_greedy.restype = ctypes.c_int
        h.sv_get_status.argtypes = [vp]
        h.sv_get_status.restype = ctypes.c_int
        h.sv_status_string.argtypes = [ctypes.c_int]
        h.sv_status_string.restype = ctypes.c_char_p
        h.sv_release.argtypes = []
        h.sv_release.restype = ctypes.c_int
        h.sv_set_launch_shape.argtypes = [i32, i32]
        h.sv_set_launch_shape.restype = ctypes.c_int
        h.sv_launch_count.argtypes = []
        h.sv_launch_count.restype = ctypes.c_uint64
        h.sv_verify_sample_noalloc.argtypes = [vp, vp, vp, vp, i64, i32, i64, i32, f32, f32, vp, vp, vp, vp]
        h.sv_verify_sample_noalloc.restype = ctypes.c_int
        h.sv_selftest_wait_timeout.argtypes = [i64, vp]
        h.sv_selftest_wait_timeout.restype = ctypes.c_int
        h.sv_verify_lookahead_sample.argtypes = [vp, vp, vp, i64, i32, i32, i64, i32, f32, vp, vp, vp, vp, vp]
        h.sv_verify_lookahead_sample.restype = ctypes.c_int
        h.sv_verify_multidraft_sample.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i32, f32, vp, vp, vp, vp, vp]
        h.sv_verify_multidraft_sample.restype = ctypes.c_int
        h.sv_set_greedy_path.argtypes = [i32]
        h.sv_set_greedy_path.restype = ctypes.c_int
        h.sv_set_sample_path.argtypes = [i32]
        h.sv_set_sample_path.restype = ctypes.c_int
        h.sv_verify_sample_lmhead.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i64, i64, f32, f32, vp, vp, vp, vp]
        h.sv_verify_sample_lmhead.restype = ctypes.c_int
        h.sv_refined_draws.argtypes = [vp]
        h.sv_refined_draws.restype = ctypes.c_int64
        h.sv_ngram_pool_bytes.argtypes = [i64, i64, i32, i32]
        h.sv_ngram_pool_bytes.restype = ctypes.c_int64
        h.sv_ngram_pool_reset.argtypes = [vp, i64, i64, i32, i32, vp]
        h.sv_ngram_pool_reset.restype = ctypes.c_int
        h.sv_ngram_pool_insert.argtypes = [vp, i64, i64, i32, i32, vp, i32, vp]
        h.sv_ngram_pool_insert.restype = ctypes.c_int
        h.sv_ngram_pool_lookup.argtypes = [vp, i64, i64, i32, i32, vp, i32, vp, vp, vp]
        h.sv_ngram_pool_lookup.restype = ctypes.c_int
        _lib_handle = h
    return _lib_handle


def exported_symbols() -> list:
    return ["sv_verify_sample", "sv_verify_greedy", "sv_get_status", "sv_status_string", "sv_release",
            "sv_set_launch_shape", "sv_launch_count", "sv_verify_sample_noalloc", "sv_selftest_wait_timeout",
            "sv_verify_lookahead_sample", "sv_verify_multidraft_sample", "sv_set_greedy_path",
            "sv_set_sample_path", "sv_ngram_pool_bytes", "sv_ngram_pool_reset", "sv_ngram_pool_insert",
            "sv_ngram_pool_lookup", "sv_refined_draws", "sv_verify_sample_lmhead"]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be torch.bfloat16 or torch.float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev_i32(a, device) -> torch.Tensor:
    """An int32 contiguous tensor on ``device`` from a tensor or an array."""
    t = a if isinstance(a, torch.Tensor) else torch.as_tensor(a)
    if t.dtype != torch.int32:
        raise TypeError(f"expected int32 token ids, got {t.dtype}")
    return _on_device(t, device, "tokens").contiguous()


def _stream_handle(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _on_device(t: torch.Tensor, device, name: str) -> torch.Tensor:
    if t.device.type == "cpu":
        return t.to(device, non_blocking=True)
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _check(t: torch.Tensor, shape, dtype, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def verify_sample(target, draft, draft_tokens, uniforms, temperature: float, top_p: float = 1.0,
                  row_stats: bool = False, out_tokens=None, out_accept_len=None, device=None):
    """Sampling-mode verify (sv_verify_sample).

    target [B,K+1,V] and draft [B,K,V] logits (bf16 or fp32), draft_tokens
    [B,K] int32, uniforms [B,K+1] fp32. Tensors on a CUDA device are used in
    place on the current stream (asynchronous). CPU tensors are copied to
    ``device`` (default: the current CUDA device), verified there, and the
    results copied back; that call returns after the results are on the host.
    Returns (out_tokens [B,K+1] int32, out_accept_len [B] int32) and, with
    ``row_stats``, a third tensor [B,2K+1,4] fp32 {m, lse, P_S, tau}.
    """
    host = target.device.type == "cpu"
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if not host:
        dev = target.device
    B, K1, V = target.shape
    K = K1 - 1
    limit = float(temperature) == 0.0
    t = _on_device(target, dev, "target")
    d = _on_device(draft, dev, "draft") if draft is not None else None
    x = _on_device(draft_tokens, dev, "draft_tokens")
    u = _on_device(uniforms, dev, "uniforms") if uniforms is not None else None
    _check(t, (B, K + 1, V), None, "target")
    dt = _dtype_code(t)
    if d is not None:
        _check(d, (B, K, V), t.dtype, "draft")
    _check(x, (B, K), torch.int32, "draft_tokens")
    if u is not None:
        _check(u, (B, K + 1), torch.float32, "uniforms")
    if not limit and (d is None or u is None):
        raise ValueError("draft and uniforms are required when temperature > 0")
    ot = torch.empty((B, K + 1), dtype=torch.int32, device=dev) if (out_tokens is None or host) else out_tokens
    oa = torch.empty((B,), dtype=torch.int32, device=dev) if (out_accept_len is None or host) else out_accept_len
    rs = torch.empty((B, 2 * K + 1, 4), dtype=torch.float32, device=dev) if row_stats else None
    with torch.cuda.device(dev):
        rc = lib().sv_verify_sample(_ptr(t), _ptr(d), _ptr(x), _ptr(u), B, K, V, dt, float(temperature),
                                    float(top_p), _ptr(ot), _ptr(oa), _ptr(rs), _stream_handle(dev))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_verify_sample")
    res = [ot, oa] + ([rs] if row_stats else [])
    if host:
        outs = [r.to("cpu", non_blocking=True) if out is None else out.copy_(r, non_blocking=True)
                for r, out in zip(res, [out_tokens, out_accept_len, None])]
        torch.cuda.current_stream(dev).synchronize()
        res = outs
    return tuple(res)


def verify_greedy(logits, cand, out_tokens=None, out_accept_len=None, best=False, device=None):
    """Greedy Lookahead verify (sv_verify_greedy).

    logits [B,G,N,V] (bf16 or fp32), cand [B,G,N-1] int32. Returns
    (out_tokens [B,N], out_accept_len [B]) and, with ``best``, the winning
    candidate [B]. CPU tensors are handled as in verify_sample.
    """
    host = logits.device.type == "cpu"
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if not host:
        dev = logits.device
    B, G, N, V = logits.shape
    lg = _on_device(logits, dev, "logits")
    c = _on_device(cand, dev, "cand")
    _check(lg, (B, G, N, V), None, "logits")
    dt = _dtype_code(lg)
    _check(c, (B, G, N - 1), torch.int32, "cand")
    ot = torch.empty((B, N), dtype=torch.int32, device=dev) if (out_tokens is None or host) else out_tokens
    oa = torch.empty((B,), dtype=torch.int32, device=dev) if (out_accept_len is None or host) else out_accept_len
    ob = torch.empty((B,), dtype=torch.int32, device=dev) if best else None
    with torch.cuda.device(dev):
        rc = lib().sv_verify_greedy(_ptr(lg), _ptr(c), B, G, N, V, dt, _ptr(ot), _ptr(oa), _ptr(ob),
                                    _stream_handle(dev))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_verify_greedy")
    res = [ot, oa] + ([ob] if best else [])
    if host:
        outs = [r.to("cpu", non_blocking=True) if out is None else out.copy_(r, non_blocking=True)
                for r, out in zip(res, [out_tokens, out_accept_len, None])]
        torch.cuda.current_stream(dev).synchronize()
        res = outs
    return tuple(res)


def verify_lookahead_sample(logits, cand, uniforms, temperature: float, out_tokens=None, out_accept_len=None,
                            best=False, row_lse=False, device=None):
    """Sampling-mode Lookahead verify of greedily produced candidates
    (sv_verify_lookahead_sample).

    logits [B,G,N,V] (bf16 or fp32), cand [B,G,N-1] int32, uniforms
    [B,(N-1)*G+1] fp32. Returns (out_tokens [B,N], out_accept_len [B]), then
    the owner of the accepted prefix [B] with ``best`` and the per-row
    log-normalisers [B,G,N] with ``row_lse``. CPU tensors are handled as in
    verify_sample.
    """
    host = logits.device.type == "cpu"
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if not host:
        dev = logits.device
    B, G, N, V = logits.shape
    lg = _on_device(logits, dev, "logits")
    c = _on_device(cand, dev, "cand")
    u = _on_device(uniforms, dev, "uniforms")
    _check(lg, (B, G, N, V), None, "logits")
    dt = _dtype_code(lg)
    _check(c, (B, G, N - 1), torch.int32, "cand")
    _check(u, (B, (N - 1) * G + 1), torch.float32, "uniforms")
    ot = torch.empty((B, N), dtype=torch.int32, device=dev) if (out_tokens is None or host) else out_tokens
    oa = torch.empty((B,), dtype=torch.int32, device=dev) if (out_accept_len is None or host) else out_accept_len
    ob = torch.empty((B,), dtype=torch.int32, device=dev) if best else None
    ol = torch.empty((B, G, N), dtype=torch.float32, device=dev) if row_lse else None
    with torch.cuda.device(dev):
        rc = lib().sv_verify_lookahead_sample(_ptr(lg), _ptr(c), _ptr(u), B, G, N, V, dt, float(temperature),
                                              _ptr(ot), _ptr(oa), _ptr(ob), _ptr(ol), _stream_handle(dev))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_verify_lookahead_sample")
    res = [ot, oa] + ([ob] if best else []) + ([ol] if row_lse else [])
    if host:
        outs = [r.to("cpu", non_blocking=True) if out is None else out.copy_(r, non_blocking=True)
                for r, out in zip(res, [out_tokens, out_accept_len, None, None])]
        torch.cuda.current_stream(dev).synchronize()
        res = outs
    return tuple(res)


def verify_multidraft_sample(target, draft, draft_tokens, uniforms, temperature: float, out_tokens=None,
                             out_accept_len=None, best=False, row_lse=False, device=None):
    """Multi-draft sampling verify (sv_verify_multidraft_sample).

    target [B,G,N,V] and draft [B,G,N-1,V] logits (bf16 or fp32), draft_tokens
    [B,G,N-1] int32, uniforms [B,(N-1)*G+1] fp32. Returns (out_tokens [B,N],
    out_accept_len [B]), then the owner [B] with ``best`` and the row
    log-normalisers [B*G*(2N-1)] (target rows, then draft rows) with
    ``row_lse``. CPU tensors are handled as in verify_sample.
    """
    host = target.device.type == "cpu"
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if not host:
        dev = target.device
    B, G, N, V = target.shape
    t = _on_device(target, dev, "target")
    d = _on_device(draft, dev, "draft")
    x = _on_device(draft_tokens, dev, "draft_tokens")
    u = _on_device(uniforms, dev, "uniforms")
    _check(t, (B, G, N, V), None, "target")
    dt = _dtype_code(t)
    _check(d, (B, G, N - 1, V), t.dtype, "draft")
    _check(x, (B, G, N - 1), torch.int32, "draft_tokens")
    _check(u, (B, (N - 1) * G + 1), torch.float32, "uniforms")
    ot = torch.empty((B, N), dtype=torch.int32, device=dev) if (out_tokens is None or host) else out_tokens
    oa = torch.empty((B,), dtype=torch.int32, device=dev) if (out_accept_len is None or host) else out_accept_len
    ob = torch.empty((B,), dtype=torch.int32, device=dev) if best else None
    ol = torch.empty((B * G * (2 * N - 1),), dtype=torch.float32, device=dev) if row_lse else None
    with torch.cuda.device(dev):
        rc = lib().sv_verify_multidraft_sample(_ptr(t), _ptr(d), _ptr(x), _ptr(u), B, G, N, V, dt,
                                               float(temperature), _ptr(ot), _ptr(oa), _ptr(ob), _ptr(ol),
                                               _stream_handle(dev))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_verify_multidraft_sample")
    res = [ot, oa] + ([ob] if best else []) + ([ol] if row_lse else [])
    if host:
        outs = [r.to("cpu", non_blocking=True) if out is None else out.copy_(r, non_blocking=True)
                for r, out in zip(res, [out_tokens, out_accept_len, None, None])]
        torch.cuda.current_stream(dev).synchronize()
        res = outs
    return tuple(res)


def get_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) its sticky device status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return lib().sv_get_status(_stream_handle(dev))


def selftest_wait_timeout(limit_ns: int = 10_000_000, device=None) -> None:
    """Enqueue the bounded-wait self-test on the current stream: a following
    get_status() reports SV_ERR_TIMEOUT (-5)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        rc = lib().sv_selftest_wait_timeout(int(limit_ns), _stream_handle(dev))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_selftest_wait_timeout")


def set_launch_shape(stages: int = 0, ctas_per_sm: int = 0) -> None:
    rc = lib().sv_set_launch_shape(stages, ctas_per_sm)
    if rc != 0:
        raise SpecVerifyError(rc, "sv_set_launch_shape")


def set_greedy_path(path: int) -> None:
    """0 (default): row argmax then match kernels; 1: the streaming kernel."""
    rc = lib().sv_set_greedy_path(int(path))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_set_greedy_path")


def set_sample_path(path: int) -> None:
    """0 (default): the row pass and the cluster decide kernel where they fit;
    1: the streaming kernel."""
    rc = lib().sv_set_sample_path(int(path))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_set_sample_path")


def launch_count() -> int:
    return int(lib().sv_launch_count())


def release() -> None:
    rc = lib().sv_release()
    if rc != 0:
        raise SpecVerifyError(rc, "sv_release")


class NgramPool:
    """The Lookahead n-gram pool in device memory (sv_ngram_pool_*): one pool
    per sequence, keyed by first token, at most ``cap`` n-grams of N tokens per
    key. ``insert`` takes int32 n-grams [B, W, N]; ``lookup`` takes the last
    generated token of each sequence [B] and returns (cand [B, G, N-1],
    count [B]) on the device, in the layout ``verify_greedy`` reads."""

    def __init__(self, B: int, V: int, N: int, cap: int, device=None):
        self.B, self.V, self.N, self.cap = B, V, N, cap
        nbytes = lib().sv_ngram_pool_bytes(B, V, N, cap)
        if nbytes < 0:
            raise SpecVerifyError(-1, "sv_ngram_pool_bytes")
        self.device = device or torch.device("cuda", torch.cuda.current_device())
        self.mem = torch.empty(max(1, int(nbytes)), dtype=torch.uint8, device=self.device)
        self.reset()

    def _stream(self):
        return ctypes.c_void_p(torch.cuda.current_stream(self.device).cuda_stream)

    def reset(self):
        rc = lib().sv_ngram_pool_reset(_ptr(self.mem), self.B, self.V, self.N, self.cap, self._stream())
        if rc != 0:
            raise SpecVerifyError(rc, "sv_ngram_pool_reset")

    def insert(self, ngrams):
        g = _dev_i32(ngrams, self.device)
        assert g.dim() == 3 and g.shape[0] == self.B and g.shape[2] == self.N
        rc = lib().sv_ngram_pool_insert(_ptr(self.mem), self.B, self.V, self.N, self.cap, _ptr(g), g.shape[1],
                                        self._stream())
        if rc != 0:
            raise SpecVerifyError(rc, "sv_ngram_pool_insert")

    def lookup(self, last, G: int, cand=None, count=None):
        """(cand [B, G, N-1], count [B]); ``cand`` and ``count`` may be given
        (int32, contiguous, on the pool's device) to be written in place."""
        t = _dev_i32(last, self.device)
        if cand is None:
            cand = torch.empty((self.B, G, self.N - 1), dtype=torch.int32, device=self.device)
        if count is None:
            count = torch.empty((self.B,), dtype=torch.int32, device=self.device)
        _check(cand, (self.B, G, self.N - 1), torch.int32, "cand")
        _check(count, (self.B,), torch.int32, "count")
        if cand.device != self.device or count.device != self.device:
            raise ValueError(f"cand and count must be on {self.device}")
        rc = lib().sv_ngram_pool_lookup(_ptr(self.mem), self.B, self.V, self.N, self.cap, _ptr(t), G, _ptr(cand),
                                        _ptr(count), self._stream())
        if rc != 0:
            raise SpecVerifyError(rc, "sv_ngram_pool_lookup")
        return cand, count


def refined_draws(device=None) -> int:
    """Draws redone in double-float so far on the current stream's scratch."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    n = lib().sv_refined_draws(_stream_handle(dev))
    if n < 0:
        raise SpecVerifyError(-3, "sv_refined_draws")
    return int(n)


def verify_sample_lmhead(h_target, h_draft, w_target, w_draft, draft_tokens, uniforms, temperature: float,
                         top_p: float = 1.0, logits: bool = False):
    """Sampling-mode verify on hidden states (sv_verify_sample_lmhead): the
    logits h · Wᵀ of the target (h_target [B,K+1,D], w_target [V,D]) and the
    draft (h_draft [B,K,D], w_draft [V,D]), all bf16 on one CUDA device, then
    the verify. Returns (out_tokens [B,K+1], out_accept_len [B]) and, with
    ``logits``, the fp32 logits [B*(K+1) + B*K, V] (target rows first)."""
    dev = h_target.device
    B, K1, D = h_target.shape
    K = K1 - 1
    V = w_target.shape[0]
    for t, name in ((h_target, "h_target"), (h_draft, "h_draft"), (w_target, "w_target"), (w_draft, "w_draft")):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != dev:
            raise TypeError(f"{name} must be a contiguous bfloat16 tensor on {dev}")
    _check(h_draft, (B, K, D), None, "h_draft")
    _check(w_draft, (V, D), None, "w_draft")
    x = _on_device(draft_tokens, dev, "draft_tokens")
    u = _on_device(uniforms, dev, "uniforms")
    out_t = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    out_a = torch.empty((B,), dtype=torch.int32, device=dev)
    lg = torch.empty((B * (K + 1) + B * K, V), dtype=torch.float32, device=dev) if logits else None
    rc = lib().sv_verify_sample_lmhead(_ptr(h_target), _ptr(h_draft), _ptr(w_target), _ptr(w_draft), _ptr(x), _ptr(u),
                                       B, K, D, V, float(temperature), float(top_p), _ptr(out_t), _ptr(out_a),
                                       _ptr(lg), _stream_handle(dev))
    if rc != 0:
        raise SpecVerifyError(rc, "sv_verify_sample_lmhead")
    return (out_t, out_a, lg) if logits else (out_t, out_a)
