"""Per-tensor weight formats.

The exporter page keeps vectors F32, embeddings and output heads F16 and the
eligible matrices Q8_0 ("rightkit-qts 0.2.3 - Qwen3-TTS 1.7B -> QTS GGUF",
section "Upstream differences & verification scope").  The library takes
16-bit matrices as f16 or bf16, embedding tables as f16 or bf16 (one
encoding for all of them), and 16-bit heads over Q8_0 matrices (tile engine).
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, assert_parity, check_parity

pytestmark = pytest.mark.gpu

WIDE_SMALL = dataclasses.replace(SMALL, code_embed_dim=SMALL.talker_hidden)


@pytest.fixture(scope="module")
def qpk():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m


def _run(qpk, g, raw, B, engines, seed=50, rows=None):
    cp = qpk.CodePredictor(g, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        P = O.Predictor.from_raw(g, raw)
        H, q0 = S.toy_inputs(g, B, seed=seed)
        rows = np.arange(B) if rows is None else rows
        for engine in engines:
            cp.set_engine(engine)
            assert_parity(check_parity(cp, P, H, q0, rows))
    finally:
        cp.close()


@pytest.mark.parametrize("B", [3, 40])
def test_all_f16(qpk, B):
    raw = S.make_weights(SMALL, seed=31, gemm_format="f16", embed_format="f16", norm_mode="perturbed")
    _run(qpk, SMALL, raw, B, ["small", "tile"])


def test_bf16_matrices_f16_heads_and_tables(qpk):
    raw = S.make_weights(SMALL, seed=32, head_format="f16", embed_format="f16", norm_mode="perturbed")
    _run(qpk, SMALL, raw, 9, ["small", "tile"])


@pytest.mark.parametrize("B", [1, 9, 140])
def test_exporter_layout(qpk, B):
    """Q8_0 matrices, f16 heads and embeddings: the tile engine streams the
    heads as 16-bit slices among the dequantised ones."""
    raw = S.make_weights(SMALL, seed=33, gemm_format="q8_0", head_format="f16", embed_format="f16",
                         norm_mode="perturbed")
    rows = None if B <= 16 else np.arange(0, B, 9)
    _run(qpk, SMALL, raw, B, ["tile"], rows=rows)


def test_exporter_layout_wide_tables(qpk):
    raw = S.make_weights(WIDE_SMALL, seed=34, gemm_format="q8_0", head_format="f16", embed_format="f16",
                         norm_mode="perturbed")
    _run(qpk, WIDE_SMALL, raw, 12, ["tile"])


@pytest.mark.parametrize("geometry,B", [("small", 6), ("wide", 3), ("full_wide", 1)])
def test_small_engine_exporter_layout(qpk, geometry, B):
    """The exporter's layout (Q8_0 matrices, f16 heads and tables; Talker-wide
    tables) on the small-batch engine: Q8_0 slices as their f16 hi + lo pair,
    16-bit head slices as they are."""
    g = {"small": SMALL, "wide": WIDE_SMALL,
         "full_wide": dataclasses.replace(S.Geometry(), code_embed_dim=S.Geometry().talker_hidden)}[geometry]
    raw = S.make_weights(g, seed=35, gemm_format="q8_0", head_format="f16", embed_format="f16",
                         norm_mode="perturbed")
    cp = qpk.CodePredictor(g, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("small")
        H, q0 = S.toy_inputs(g, B, seed=2)
        assert_parity(check_parity(cp, O.Predictor.from_raw(g, raw), H, q0, np.arange(B)))
    finally:
        cp.close()


def _load_status(qpk, raw):
    cp = qpk.CodePredictor(SMALL, max_batch=2)
    try:
        cp.load_raw_weights(raw)
        return 0
    except qpk.QpError as e:
        return e.code
    finally:
        cp.close()


def test_loader_refusals(qpk):
    dtype_err = {v: k for k, v in qpk.STATUS_NAMES.items()}["QP_ERR_WEIGHT_DTYPE"]
    # embedding tables in two encodings
    raw = S.make_weights(SMALL, seed=36)
    t = raw["code_pred.codec_embd.3.weight"]
    raw["code_pred.codec_embd.3.weight"] = S.RawTensor(t.name, "f16", t.shape,
                                                       O.bf16_to_f32(t.data).reshape(t.shape).astype(np.float16))
    assert _load_status(qpk, raw) == dtype_err
    # Q8_0 heads over 16-bit matrices
    raw = S.make_weights(SMALL, seed=37, head_format="q8_0")
    assert _load_status(qpk, raw) == dtype_err
    # matrices of one role in two formats
    raw = S.make_weights(SMALL, seed=38)
    q8 = S.make_weights(SMALL, seed=38, gemm_format="q8_0")
    raw["code_pred.blk.1.ffn_up.weight"] = q8["code_pred.blk.1.ffn_up.weight"]
    assert _load_status(qpk, raw) == dtype_err
