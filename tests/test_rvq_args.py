"""Host-side argument checks of include/qp_rvq.h: every rejected call returns
QP_ERR_ARG before touching the device, so these run without a GPU."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def lib():
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m.lib()


FAKE = 0x1000            # 16-byte aligned; never dereferenced by a rejected call


def test_decode_rejects_bad_arguments(lib):
    d = lib.qp_rvq_decode
    assert d(FAKE, 16, 2048, 6, FAKE, 10, FAKE, None, None) == 1        # dim not a multiple of 4
    assert d(FAKE, 33, 2048, 8, FAKE, 10, FAKE, None, None) == 1        # more than 32 codebooks
    assert d(FAKE, 0, 2048, 8, FAKE, 10, FAKE, None, None) == 1         # no codebooks
    assert d(FAKE, 4, 0, 8, FAKE, 10, FAKE, None, None) == 1            # empty codebooks
    assert d(FAKE, 4, 16, 8, FAKE, -1, FAKE, None, None) == 1           # negative frame count
    assert d(None, 4, 16, 8, FAKE, 3, FAKE, None, None) == 1            # null codebooks
    assert d(FAKE + 4, 4, 16, 8, FAKE, 3, FAKE, None, None) == 1        # misaligned codebooks
    assert d(FAKE, 4, 16, 8, FAKE + 2, 3, FAKE, None, None) == 1        # misaligned codes
    assert d(FAKE, 4, 16, 8, FAKE, 0, FAKE, None, None) == 0            # nothing to do


def test_normalize_rejects_bad_arguments(lib):
    n = lib.qp_rvq_normalize
    assert n(FAKE, FAKE, 16, 2048, 10, FAKE, None) == 1                 # dim not a multiple of 4
    assert n(None, FAKE, 16, 2048, 8, FAKE, None) == 1
    assert n(FAKE, FAKE, 16, 2048, 8, None, None) == 1
    assert n(FAKE, FAKE, 0, 2048, 8, FAKE, None) == 1
    assert n(FAKE + 8, FAKE, 1, 1, 4, FAKE, None) == 1                  # misaligned embedding_sum
