"""The C-ABI library loads and exports every entry point include/qp.h declares.

These run without a GPU: only calls that fail argument checks before any
CUDA call are made.
"""
import ctypes
import glob
import os
import re

import pytest

import codebook_rvq_code_gb300 as qpk
from codebook_rvq_code_gb300 import build as qb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qb.build()
    return qpk.load_library()


def declared_functions():
    names = set()
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(qp_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(qpk.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.qp_abi_version() == 1
    for code in range(12):
        assert lib.qp_status_string(code)
    assert lib.qp_status_string(999) == b"unknown status"


def test_default_geometry_is_the_1p7b_predictor(lib):
    g = qpk.default_geometry()
    assert (g.hidden, g.layers, g.n_q_heads, g.n_kv_heads, g.head_dim, g.ffn) == (1024, 5, 16, 8, 128, 3072)
    assert (g.vocab, g.n_steps, g.talker_hidden, g.code_embed_dim, g.q0_vocab) == (2048, 15, 2048, 1024, 2048)
    assert g.rms_eps == pytest.approx(1e-6) and g.rope_theta == pytest.approx(1e6)
    assert lib.qp_default_geometry(None) == 1


def test_create_rejects_bad_arguments_before_touching_cuda(lib):
    h = ctypes.c_void_p()
    g = qpk.default_geometry()
    assert lib.qp_create(None, 1, ctypes.byref(h)) == 1
    assert lib.qp_create(ctypes.byref(g), 0, ctypes.byref(h)) == 1
    assert lib.qp_create(ctypes.byref(g), 1 << 20, ctypes.byref(h)) == 1
    for field, bad in (("head_dim", 64), ("n_q_heads", 12), ("hidden", 1000), ("n_steps", 16),
                       ("code_embed_dim", 1536), ("vocab", 100)):
        gg = qpk.default_geometry()
        setattr(gg, field, bad)
        assert lib.qp_create(ctypes.byref(gg), 1, ctypes.byref(h)) == 1, field
        assert h.value is None


def test_null_handle_calls_are_rejected(lib):
    assert lib.qp_load_weights(None, None, 0, None) == 1
    assert lib.qp_predict_frames(None, 1, None, None, None, None, None) == 1
    assert lib.qp_predict_frames_ex(None, 1, None, None, None, None, None, None, None) == 1
    assert lib.qp_predict_frames_host(None, 1, None, None, None, None, None) == 1
    assert lib.qp_get_device_status(None, None) == 1
    assert lib.qp_launches_per_call(None, 1, 0) == -1
    lib.qp_destroy(None)


def test_product_package_has_no_cpu_path():
    """The binding loads only libqp.so; a missing library is an ImportError."""
    with pytest.raises(ImportError):
        qpk.load_library("/nonexistent/libqp.so")
    src = open(os.path.join(ROOT, "codebook_rvq_code_gb300", "__init__.py")).read()
    assert "oracle" not in src
