"""The CPU oracle of the sampling verify on LM-head logits (h · W^T in fp64),
the computation a fused LM-head GEMM with a verify epilogue reproduces: it is
the pinned sampling-mode oracle applied to exact products (no GPU)."""
import pytest

import oracle
import specgen as sg

from pins import check_lmhead_identity, check_lmhead_integer_products


@pytest.fixture(scope="module")
def lib():
    return oracle._lib()


def test_identity_heads(lib):
    check_lmhead_identity(lib)


@pytest.mark.parametrize("dtype", [sg.F32, sg.BF16])
def test_integer_products(lib, dtype):
    check_lmhead_integer_products(lib, dtype)
