"""The oracle's n-gram pool ("Lookahead Decoding 完全拆解", section "N-gram 池与
身份判定") against hand-worked cases and the properties the page fixes."""
import pytest

import oracle
from pins import check_ngram_golden, check_ngram_properties


@pytest.fixture(scope="module")
def lib():
    return oracle._lib()


def test_ngram_golden(lib):
    check_ngram_golden(lib)


def test_ngram_properties(lib):
    check_ngram_properties(lib)
