"""Weights loaded from GGUF files (include/qp_gguf.h) run the predictor like
the same weights handed over directly, and match the oracle."""
import dataclasses

import numpy as np
import pytest

import oracle as O
import synthetic as S
from synthetic import gguf as SG
from _parity import SMALL, assert_parity, check_parity, decided_prefix, run_gpu

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


@pytest.mark.parametrize("g", [SMALL, WIDE_SMALL])
def test_gguf_exporter_layout(qpk, tmp_path, g):
    raw = S.make_weights(g, seed=61, gemm_format="q8_0", head_format="f16", embed_format="f16",
                         norm_mode="perturbed")
    pred, talk = str(tmp_path / "p.gguf"), str(tmp_path / "t.gguf")
    SG.write_predictor_files(pred, talk, g, raw)
    P, T = qpk.GgufFile(pred), qpk.GgufFile(talk)
    geo = P.geometry(T)
    B = 20
    a = qpk.CodePredictor(geo, max_batch=B)
    b = qpk.CodePredictor(g, max_batch=B)
    try:
        a.load_gguf(P, T)
        b.load_raw_weights(raw)
        H, q0 = S.toy_inputs(g, B, seed=8)
        assert_parity(check_parity(a, O.Predictor.from_raw(g, raw), H, q0, np.arange(0, B, 3)))
        ca, la = run_gpu(a, H, q0)
        cb, lb = run_gpu(b, H, q0)
        cm, lm = decided_prefix(la, lb)
        np.testing.assert_array_equal(ca[cm], cb[cm])
        np.testing.assert_allclose(la[lm], lb[lm], rtol=0, atol=1e-3)
    finally:
        a.close()
        b.close()


def test_gguf_missing_tensor(qpk, tmp_path):
    raw = S.make_weights(SMALL, seed=62)
    del raw["code_pred.blk.1.attn_k_norm.weight"]
    pred, talk = str(tmp_path / "p.gguf"), str(tmp_path / "t.gguf")
    SG.write_predictor_files(pred, talk, SMALL, raw)
    cp = qpk.CodePredictor(SMALL, max_batch=2)
    try:
        with pytest.raises(qpk.QpError) as e:
            cp.load_gguf(pred, talk)
        assert e.value.code == 3   # QP_ERR_WEIGHT_MISSING
    finally:
        cp.close()
