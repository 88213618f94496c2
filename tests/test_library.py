"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side argument checks reject bad calls before any launch. No
GPU is needed: every call here fails its checks before touching CUDA."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_39_gb300 as svpkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    svpkg.build()
    return svpkg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "sv_verify_sample" in names and "sv_verify_greedy" in names
    assert set(names) == set(svpkg.exported_symbols())


def test_library_exports_every_declared_symbol(lib):
    out = os.popen(f"nm -D --defined-only {svpkg._SO}").read()
    exported = set(re.findall(r" T (sv_[a-z_]+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for rc in range(-6, 1):
        assert lib.sv_status_string(rc)
    assert lib.sv_status_string(0) == b"ok"


def test_host_argument_checks(lib):
    f = lib.sv_verify_sample
    p = ctypes.c_void_p(16)  # never dereferenced: the checks fail first
    # dtype
    assert f(p, p, p, p, 4, 3, 100, 7, 1.0, 1.0, p, p, None, None) == -2
    # shapes
    assert f(p, p, p, p, -1, 3, 100, 1, 1.0, 1.0, p, p, None, None) == -1
    assert f(p, p, p, p, 4, 0, 100, 1, 1.0, 1.0, p, p, None, None) == -1
    assert f(p, p, p, p, 4, 3, 1, 1, 1.0, 1.0, p, p, None, None) == -1
    assert f(p, p, p, p, 4, 3, 1 << 31, 1, 1.0, 1.0, p, p, None, None) == -1
    # temperature / top_p
    assert f(p, p, p, p, 4, 3, 100, 1, -0.5, 1.0, p, p, None, None) == -1
    assert f(p, p, p, p, 4, 3, 100, 1, float("nan"), 1.0, p, p, None, None) == -1
    assert f(p, p, p, p, 4, 3, 100, 1, 1.0, 0.0, p, p, None, None) == -1
    assert f(p, p, p, p, 4, 3, 100, 1, 1.0, 1.5, p, p, None, None) == -1
    # null pointers
    assert f(None, p, p, p, 4, 3, 100, 1, 1.0, 1.0, p, p, None, None) == -1
    assert f(p, None, p, p, 4, 3, 100, 1, 1.0, 1.0, p, p, None, None) == -1
    assert f(p, p, p, None, 4, 3, 100, 1, 1.0, 1.0, p, p, None, None) == -1
    # misaligned logits for the dtype
    q = ctypes.c_void_p(17)
    assert f(q, p, p, p, 4, 3, 100, 1, 1.0, 1.0, p, p, None, None) == -2
    # B == 0 is a no-op, even with null pointers
    assert f(None, None, None, None, 0, 3, 100, 1, 1.0, 1.0, None, None, None, None) == 0
    g = lib.sv_verify_greedy
    assert g(p, p, 4, 0, 5, 100, 1, p, p, None, None) == -1
    assert g(p, p, 4, 7, 1, 100, 1, p, p, None, None) == -1
    assert g(p, p, 4, 7, 5, 100, 9, p, p, None, None) == -2
    assert g(None, None, 0, 7, 5, 100, 1, None, None, None, None) == 0
    la = lib.sv_verify_lookahead_sample
    assert la(p, p, p, 4, 7, 5, 100, 9, 1.0, p, p, None, None, None) == -2
    assert la(p, p, p, 4, 0, 5, 100, 1, 1.0, p, p, None, None, None) == -1    # G < 1
    assert la(p, p, p, 4, 33, 2, 100, 1, 1.0, p, p, None, None, None) == -1   # G > 32
    assert la(p, p, p, 4, 7, 1, 100, 1, 1.0, p, p, None, None, None) == -1    # N < 2
    assert la(p, p, p, 4, 16, 65, 100, 1, 1.0, p, p, None, None, None) == -1  # G*N > 1024
    assert la(p, p, p, 4, 32, 6, 100, 1, 1.0, p, p, None, None, None) == -1   # G*G*(N-1) > 4096
    assert la(p, p, p, 4, 7, 5, 1, 1, 1.0, p, p, None, None, None) == -1      # V < 2
    assert la(p, p, p, 1 << 40, 7, 5, 100, 1, 1.0, p, p, None, None, None) == -1
    assert la(p, p, p, 4, 7, 5, 100, 1, 0.0, p, p, None, None, None) == -1    # T = 0
    assert la(p, p, p, 4, 7, 5, 100, 1, float("inf"), p, p, None, None, None) == -1
    assert la(p, p, None, 4, 7, 5, 100, 1, 1.0, p, p, None, None, None) == -1  # no uniforms
    assert la(q, p, p, 4, 7, 5, 100, 1, 1.0, p, p, None, None, None) == -2    # misaligned bf16 logits
    assert la(None, None, None, 0, 7, 5, 100, 1, 1.0, None, None, None, None, None) == 0
    md = lib.sv_verify_multidraft_sample
    assert md(p, p, p, p, 4, 7, 5, 100, 9, 1.0, p, p, None, None, None) == -2
    assert md(p, p, p, p, 4, 33, 2, 100, 1, 1.0, p, p, None, None, None) == -1   # G > 32
    assert md(p, p, p, p, 4, 16, 10, 100, 1, 1.0, p, p, None, None, None) == -1  # G*G*(N-1) > 2048
    assert md(p, p, p, p, 4, 7, 1, 100, 1, 1.0, p, p, None, None, None) == -1    # N < 2
    assert md(p, p, p, p, 4, 7, 5, 100, 1, 0.0, p, p, None, None, None) == -1    # T = 0
    assert md(p, None, p, p, 4, 7, 5, 100, 1, 1.0, p, p, None, None, None) == -1  # no draft
    assert md(p, q, p, p, 4, 7, 5, 100, 1, 1.0, p, p, None, None, None) == -2    # misaligned draft
    assert md(None, None, None, None, 0, 7, 5, 100, 1, 1.0, None, None, None, None, None) == 0
    # the verify on hidden states: its argument checks come before any device work
    lm = lib.sv_verify_sample_lmhead
    assert lm(p, p, p, p, p, p, 2, 1, 100, 50, 1.0, 1.0, p, p, None, None) == -1       # D not a multiple of 64
    assert lm(p, p, p, p, p, p, 2, 1, 64, 50, 0.0, 1.0, p, p, None, None) == -1        # T = 0
    assert lm(p, p, p, p, p, p, 2, 1, 64, 50, 1.0, 0.0, p, p, None, None) == -1        # top_p = 0
    assert lm(p, p, p, p, p, p, 2, 0, 64, 50, 1.0, 1.0, p, p, None, None) == -1        # K < 1
    assert lm(p, p, p, p, p, p, 2, 1, 64, 1, 1.0, 1.0, p, p, None, None) == -1         # V < 2
    assert lm(p, p, p, p, p, p, 1 << 30, 1, 64, 50, 1.0, 1.0, p, p, None, None) == -1  # B(2K+1) >= 2^31
    assert lm(None, p, p, p, p, p, 2, 1, 64, 50, 1.0, 1.0, p, p, None, None) == -1     # no target states
    assert lm(p, p, p, None, p, p, 2, 1, 64, 50, 1.0, 1.0, p, p, None, None) == -1     # no draft head
    assert lm(q, p, p, p, p, p, 2, 1, 64, 50, 1.0, 1.0, p, p, None, None) == -2        # misaligned states
    assert lm(None, None, None, None, None, None, 0, 1, 64, 50, 1.0, 1.0, None, None, None, None) == 0
    assert lib.sv_set_greedy_path(2) == -1 and lib.sv_set_greedy_path(-1) == -1
    assert lib.sv_set_launch_shape(7, 1) == -1
    assert lib.sv_set_launch_shape(0, 0) == 0
    # the wait self-test checks its limit before touching the device
    assert lib.sv_selftest_wait_timeout(-1, None) == -1
    assert lib.sv_selftest_wait_timeout(3_000_000_000, None) == -1


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(svpkg, "_SO", str(tmp_path / "missing.so"))
    monkeypatch.setattr(svpkg, "_lib_handle", None)
    with pytest.raises(RuntimeError):
        svpkg.lib()
