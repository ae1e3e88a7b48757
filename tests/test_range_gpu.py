"""Parity at large activation magnitudes (f16 operand range).

The tensor cores take f16 operands, whose largest finite value is 65504.
The operand rows built from the residual stream, x * w_norm before the
RMSNorm's 1/RMS, and from the Talker state H, scale with the inputs.  Here H
is scaled by 1e2 and 1e4 and the layers' attn_norm / ffn_norm weights are
drawn log-uniform up to x30, which puts those rows far above 65504.  Each
engine must still match the oracle under the usual rules (logits within
3e-2, decidable codes exact).  The oracle is in f32 and needs no scaling.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, assert_parity, check_parity, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qpk():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m


@pytest.fixture(scope="module")
def full_wide(qpk):
    g = S.Geometry()
    raw = S.make_weights(g, seed=0, norm_mode="wide")
    cp = qpk.CodePredictor(g, max_batch=32)
    cp.load_raw_weights(raw)
    yield g, O.Predictor.from_raw(g, raw), cp
    cp.close()


@pytest.mark.parametrize("engine", ["small", "tile"])
@pytest.mark.parametrize("hscale", [1e2, 1e4])
@pytest.mark.parametrize("B", [1, 8])
def test_full_geometry_bf16_large_magnitudes(full_wide, engine, hscale, B):
    """Configuration 1's recipe (at B = 1, and at 8 frames), H x hscale."""
    g, P, cp = full_wide
    w = S.make_workload(1, g, B=B)
    H = (w.H * np.float32(hscale)).astype(np.float32)
    cp.set_engine(engine)
    try:
        st = check_parity(cp, P, H, w.q0, sample_rows(B, 4))
    finally:
        cp.set_engine("auto")
    print(engine, hscale, B, st)
    assert_parity(st)


@pytest.mark.parametrize("hscale", [1e2, 1e4])
def test_full_geometry_q8_0_large_magnitudes(qpk, hscale):
    """Configuration 5 (every GEMM matrix Q8_0, 1024 frames), H x hscale,
    wide norms; sampled frames against the oracle on exact d*q weights."""
    g = S.Geometry()
    w = S.make_workload(5, g)
    raw = S.make_weights(g, seed=w.weight_seed, gemm_format=w.gemm_format, norm_mode="wide")
    P = O.Predictor.from_raw(g, raw)
    cp = qpk.CodePredictor(g, max_batch=w.B)
    try:
        cp.load_raw_weights(raw)
        H = (w.H * np.float32(hscale)).astype(np.float32)
        st = check_parity(cp, P, H, w.q0, sample_rows(w.B, 6))
    finally:
        cp.close()
    print("q8_0", hscale, st)
    assert_parity(st)


@pytest.mark.parametrize("engine", ["small", "tile"])
@pytest.mark.parametrize("hscale", [1e4, 1e6])
def test_small_geometry_large_magnitudes_all_rows(qpk, engine, hscale):
    """Every frame of a small geometry at ragged B, H up to x1e6 (f16(H)
    alone would overflow), wide norms, both engines."""
    raw = S.make_weights(SMALL, seed=21, norm_mode="wide")
    P = O.Predictor.from_raw(SMALL, raw)
    cp = qpk.CodePredictor(SMALL, max_batch=33)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine(engine)
        H, q0 = S.toy_inputs(SMALL, 33, seed=5)
        H = (H * np.float32(hscale)).astype(np.float32)
        st = check_parity(cp, P, H, q0, np.arange(33))
    finally:
        cp.close()
    print(engine, hscale, st)
    assert_parity(st)
