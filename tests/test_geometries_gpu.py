"""Hidden sizes between the tested ones, through the C ABI, against the
oracle: every multiple of 128 is accepted, so 384 (three 128-row tiles) and
768 (six; operand builds whose 8-column chunks do not fill whole warps per
row half) run on the tile and small-batch engines and under the automatic
choice.  The cluster engine's operand build needs a row half of 256 or 512
columns (hidden 512 or 1024): it refuses 768, and the automatic choice
serves that geometry on another engine.
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, assert_parity, check_parity, sample_rows

pytestmark = pytest.mark.gpu

H384 = dataclasses.replace(SMALL, hidden=384, code_embed_dim=384, ffn=640, vocab=384)
H768 = dataclasses.replace(SMALL, hidden=768, code_embed_dim=768, ffn=768, vocab=512, talker_hidden=512)


@pytest.fixture(scope="module")
def qpk():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m


@pytest.mark.parametrize("geo", ["h384", "h768"])
@pytest.mark.parametrize("engine,B", [("tile", 5), ("small", 5), ("small", 33), ("auto", 3), ("auto", 26)])
def test_hidden_sizes_each_engine(qpk, geo, engine, B):
    g = {"h384": H384, "h768": H768}[geo]
    raw = S.make_weights(g, seed=61, norm_mode="perturbed")
    cp = qpk.CodePredictor(g, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine(engine)
        H, q0 = S.toy_inputs(g, B, seed=62 + B)
        assert_parity(check_parity(cp, O.Predictor.from_raw(g, raw), H, q0, sample_rows(B, 6)))
    finally:
        cp.close()


def test_cluster_engine_refuses_hidden_768(qpk):
    import torch
    raw = S.make_weights(H768, seed=63)
    cp = qpk.CodePredictor(H768, max_batch=4)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(H768, 4, seed=64)
        with pytest.raises(qpk.QpError) as e:
            cp.predict(torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda())
        assert e.value.code == 1
    finally:
        cp.close()
