"""GGUF reading (include/qp_gguf.h) on the host: the tensor table, the
geometry from the exporter's keys and tensor shapes, and refusals of
malformed files.  No CUDA call is made."""
import dataclasses
import os

import numpy as np
import pytest

import synthetic as S
from synthetic import gguf as SG
from _parity import SMALL

WIDE_SMALL = dataclasses.replace(SMALL, code_embed_dim=SMALL.talker_hidden)


@pytest.fixture(scope="module")
def qpk():
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m


def _files(tmp_path, g, raw, alignment=32):
    pred, talk = str(tmp_path / "predictor.gguf"), str(tmp_path / "talker.gguf")
    SG.write_predictor_files(pred, talk, g, raw, alignment=alignment)
    return pred, talk


@pytest.mark.parametrize("g,alignment", [(SMALL, 32), (WIDE_SMALL, 64)])
def test_table_and_geometry(qpk, tmp_path, g, alignment):
    raw = S.make_weights(g, seed=3, gemm_format="q8_0", head_format="f16", embed_format="f16")
    pred, talk = _files(tmp_path, g, raw, alignment)
    P, T = qpk.GgufFile(pred), qpk.GgufFile(talk)
    table = P.tensors()
    assert len(table) == 3 + 11 * g.layers + 2 * g.n_steps   # 88 for the 1.7B geometry
    for name, dt, shape in table:
        t = raw[name]
        assert dt == t.dtype, name
        assert shape == (t.shape[0], t.shape[1] if len(t.shape) > 1 else 0), name
    assert [n for n, _, _ in T.tensors()] == ["talker.codec_embd.weight", "talker.output_norm.weight"]
    got = P.geometry(T)
    for f in ("hidden", "layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "n_steps",
              "talker_hidden", "code_embed_dim", "q0_vocab"):
        assert getattr(got, f) == getattr(g, f), f
    assert got.rms_eps == pytest.approx(g.rms_eps) and got.rope_theta == pytest.approx(g.rope_theta)


def test_geometry_needs_the_q0_table(qpk, tmp_path):
    raw = S.make_weights(SMALL, seed=4)
    pred, talk = _files(tmp_path, SMALL, raw)
    with pytest.raises(qpk.QpError) as e:
        qpk.GgufFile(pred).geometry()
    assert e.value.code == 3   # QP_ERR_WEIGHT_MISSING


def test_malformed_files_are_refused(qpk, tmp_path):
    raw = S.make_weights(SMALL, seed=5)
    pred, _ = _files(tmp_path, SMALL, raw)
    data = open(pred, "rb").read()
    bad = tmp_path / "bad.gguf"
    cases = {
        "magic": b"GGUX" + data[4:],
        "version": data[:4] + (9).to_bytes(4, "little") + data[8:],
        "truncated table": data[:200],
        "data past the end": data[:-64],
    }
    for what, blob in cases.items():
        bad.write_bytes(blob)
        with pytest.raises(qpk.QpError):
            qpk.GgufFile(str(bad))
    with pytest.raises(qpk.QpError):
        qpk.GgufFile(str(tmp_path / "missing.gguf"))
    assert os.path.exists(pred)
