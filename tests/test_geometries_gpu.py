"""Geometries the C ABI accepts beyond the tested predictor shapes, against
the oracle: hidden sizes of 384 (three 128-row tiles), 768 (six; operand
builds whose 8-column chunks do not fill whole warps per row half) and 2048,
and one or four q heads per kv head, on the tile and small-batch engines
and under the automatic choice.  The cluster engine's operand build needs a row half of 256 or 512
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
# other ratios of q heads to kv heads than the predictor's 2 (one, and four), and a wide stream
MHA = dataclasses.replace(SMALL, n_q_heads=2, n_kv_heads=2)
GQA4 = dataclasses.replace(SMALL, n_q_heads=8, n_kv_heads=2)
H2048 = dataclasses.replace(SMALL, hidden=2048, code_embed_dim=2048, layers=1, ffn=1024)
GEOS = {"h384": H384, "h768": H768, "mha": MHA, "gqa4": GQA4, "h2048": H2048}


@pytest.fixture(scope="module")
def qpk():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m


@pytest.mark.parametrize("geo", list(GEOS))
@pytest.mark.parametrize("engine,B", [("tile", 5), ("small", 5), ("small", 33), ("auto", 3), ("auto", 26)])
def test_hidden_sizes_each_engine(qpk, geo, engine, B):
    g = GEOS[geo]
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


@pytest.mark.parametrize("n_steps", [1, 7])
def test_cluster_engine_fewer_steps(qpk, n_steps):
    """A loop shorter than 15 steps on the cluster engine (its KV cache keeps
    16 positions per layer whatever the step count)."""
    from test_cluster_gpu import CL
    g = dataclasses.replace(CL, n_steps=n_steps)
    raw = S.make_weights(g, seed=65, norm_mode="perturbed")
    cp = qpk.CodePredictor(g, max_batch=25)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        for B in (3, 25):
            H, q0 = S.toy_inputs(g, B, seed=66 + B)
            assert_parity(check_parity(cp, O.Predictor.from_raw(g, raw), H, q0, sample_rows(B, 5)))
    finally:
        cp.close()
