"""Talker-wide code tables: every step's input passes through small_to_mtp.

The exporter page gives the predictor's 15 code-embedding tables as
2048 x 2048 ("rightkit-qts 0.2.3 - Qwen3-TTS 1.7B -> QTS GGUF", section
"Expected verification shapes"), twice the stream's width, so a step's input
E[k-2][q_{k-1}] is projected like H and E0[q0] (the oracle's reading,
pinned in test_oracle_pins.py).  Both engines serve this geometry with a
projection GEMM per step.
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, assert_parity, check_parity

pytestmark = pytest.mark.gpu

WIDE_SMALL = dataclasses.replace(SMALL, code_embed_dim=SMALL.talker_hidden)
WIDE_FULL = dataclasses.replace(S.Geometry(), code_embed_dim=S.Geometry().talker_hidden)


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
def wide(qpk):
    raw = S.make_weights(WIDE_SMALL, seed=21, norm_mode="perturbed")
    cp = qpk.CodePredictor(WIDE_SMALL, max_batch=64)
    cp.load_raw_weights(raw)
    yield raw, O.Predictor.from_raw(WIDE_SMALL, raw), cp
    cp.close()


@pytest.mark.parametrize("engine", ["small", "tile"])
@pytest.mark.parametrize("B", [1, 2, 5, 8, 9, 32, 64])
def test_wide_tables_match_the_oracle(wide, engine, B):
    raw, P, cp = wide
    cp.set_engine(engine)
    try:
        H, q0 = S.toy_inputs(WIDE_SMALL, B, seed=300 + B)
        assert_parity(check_parity(cp, P, H, q0, np.arange(B)))
    finally:
        cp.set_engine("auto")


def test_wide_tables_sampling(wide):
    raw, P, cp = wide
    B, T, k = 6, 0.9, 20
    H, q0 = S.toy_inputs(WIDE_SMALL, B, seed=41)
    gum = S.gumbel_noise((B, WIDE_SMALL.n_steps, WIDE_SMALL.vocab), seed=3)
    assert_parity(check_parity(cp, P, H, q0, np.arange(B), T, k, gum))


def test_wide_tables_q8_0_and_more_frames(qpk):
    """Q8_0 matrices (the exporter's format for eligible matrices) and 150
    frames (two 128-row chunks): the tile engine."""
    raw = S.make_weights(WIDE_SMALL, seed=7, gemm_format="q8_0", norm_mode="perturbed")
    cp = qpk.CodePredictor(WIDE_SMALL, max_batch=150)
    try:
        cp.load_raw_weights(raw)
        H, q0 = S.toy_inputs(WIDE_SMALL, 150, seed=17)
        rows = np.arange(0, 150, 7)
        assert_parity(check_parity(cp, O.Predictor.from_raw(WIDE_SMALL, raw), H, q0, rows))
    finally:
        cp.close()


def test_wide_tables_feedback_embeddings(wide):
    import torch
    raw, P, cp = wide
    codes = np.random.default_rng(5).integers(0, WIDE_SMALL.vocab, size=(7, WIDE_SMALL.n_steps)).astype(np.int32)
    got = cp.code_embeddings(torch.from_numpy(codes).cuda()).cpu().numpy()
    assert got.shape == (7, WIDE_SMALL.n_steps, WIDE_SMALL.code_embed_dim)
    np.testing.assert_array_equal(got, O.code_embeddings(P, codes))


def test_wide_tables_full_geometry(qpk):
    """The 1.7B geometry with 2048-wide tables, 4 frames against the oracle."""
    raw = S.make_weights(WIDE_FULL, seed=0)
    cp = qpk.CodePredictor(WIDE_FULL, max_batch=4)
    try:
        cp.load_raw_weights(raw)
        H, q0 = S.toy_inputs(WIDE_FULL, 4, seed=8)
        P = O.Predictor.from_raw(WIDE_FULL, raw)
        for engine in ("small", "tile"):
            cp.set_engine(engine)
            assert_parity(check_parity(cp, P, H, q0, np.arange(4)))
    finally:
        cp.close()
