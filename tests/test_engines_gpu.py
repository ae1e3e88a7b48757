"""Both schedules of the frame loop against the oracle, through the C ABI.

The small-batch engine serves bf16 calls of at most 64 frames (the default
for them up to 40); the tile engine serves every call.  Each is forced here on the
batch sizes the other would take, and the two are compared with each other.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, TOL, assert_parity, check_parity, decided_prefix, run_gpu, sample_rows

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
def small(qpk):
    raw = S.make_weights(SMALL, seed=11, norm_mode="perturbed")
    cp = qpk.CodePredictor(SMALL, max_batch=96)
    cp.load_raw_weights(raw)
    yield raw, O.Predictor.from_raw(SMALL, raw), cp
    cp.set_engine("auto")
    cp.close()


@pytest.mark.parametrize("engine", ["small", "tile"])
@pytest.mark.parametrize("B", [1, 2, 7, 8, 9, 31, 64])
def test_small_geometry_each_engine(small, engine, B):
    raw, P, cp = small
    cp.set_engine(engine)
    try:
        H, q0 = S.toy_inputs(SMALL, B, seed=100 + B)
        assert_parity(check_parity(cp, P, H, q0, np.arange(B)))
    finally:
        cp.set_engine("auto")


@pytest.mark.parametrize("engine", ["small", "tile"])
def test_small_geometry_sampling_each_engine(small, engine):
    raw, P, cp = small
    cp.set_engine(engine)
    try:
        B = 19
        H, q0 = S.toy_inputs(SMALL, B, seed=23)
        gum = S.gumbel_noise((B, SMALL.n_steps, SMALL.vocab), seed=24)
        assert_parity(check_parity(cp, P, H, q0, np.arange(B), 0.8, 12, gum))
    finally:
        cp.set_engine("auto")


def test_engines_agree(small):
    raw, P, cp = small
    H, q0 = S.toy_inputs(SMALL, 40, seed=31)
    cp.set_engine("small")
    try:
        a = run_gpu(cp, H, q0)
        cp.set_engine("tile")
        b = run_gpu(cp, H, q0)
    finally:
        cp.set_engine("auto")
    cm, lm = decided_prefix(a[1], b[1])
    np.testing.assert_array_equal(a[0][cm], b[0][cm])
    np.testing.assert_allclose(a[1][lm], b[1][lm], rtol=0, atol=5e-3)


def test_small_refuses_what_it_cannot_serve(small, qpk):
    import torch
    raw, P, cp = small
    cp.set_engine("small")
    try:
        H = torch.zeros((65, SMALL.talker_hidden), device="cuda")
        q0 = torch.zeros(65, dtype=torch.int32, device="cuda")
        with pytest.raises(qpk.QpError) as e:
            cp.predict(H, q0)                 # more than 64 frames
        assert e.value.code == 1
        cp.predict(H[:64], q0[:64])           # 64 is served
        torch.cuda.synchronize()
        assert cp.device_status() == 0
    finally:
        cp.set_engine("auto")
    assert cp._lib.qp_set_engine(cp._h, 7) == 1   # unknown engine: QP_ERR_ARG


@pytest.mark.parametrize("B", [1, 5, 33])
def test_small_engine_serves_q8_0(qpk, B):
    """Q8_0 matrices on the small-batch engine, through the exact f16 pair
    hi + lo packed at load time: every frame against the oracle's exact d*q
    weights, and the two engines on the same handle agree."""
    raw = S.make_weights(SMALL, seed=12, gemm_format="q8_0", norm_mode="perturbed")
    P = O.Predictor.from_raw(SMALL, raw)
    cp = qpk.CodePredictor(SMALL, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        H, q0 = S.toy_inputs(SMALL, B, seed=60 + B)
        cp.set_engine("small")
        assert_parity(check_parity(cp, P, H, q0, np.arange(B)))
        _, l_small = run_gpu(cp, H, q0)
        cp.set_engine("tile")
        _, l_tile = run_gpu(cp, H, q0)
        _, lmask = decided_prefix(l_small, l_tile)
        assert np.abs(l_small - l_tile)[lmask].max() <= TOL
    finally:
        cp.close()


@pytest.fixture(scope="module")
def full_bf16(qpk):
    g = S.Geometry()
    raw = S.make_weights(g, seed=0)
    cp = qpk.CodePredictor(g, max_batch=64)
    cp.load_raw_weights(raw)
    yield g, raw, O.Predictor.from_raw(g, raw), cp
    cp.close()


@pytest.mark.parametrize("engine", ["small", "tile"])
@pytest.mark.parametrize("cfg,max_rows", [(1, 1), (2, 12)])
def test_full_size_small_batch_each_engine(full_bf16, engine, cfg, max_rows):
    g, raw, P, cp = full_bf16
    w = S.make_workload(cfg, g)
    cp.set_engine(engine)
    try:
        st = check_parity(cp, P, w.H, w.q0, sample_rows(w.B, max_rows), w.temperature, w.top_k, w.gumbel)
    finally:
        cp.set_engine("auto")
    print(engine, cfg, st)
    assert_parity(st)


def test_full_size_sampling_small(full_bf16):
    """Configuration 4's sampling parameters at a batch the small-batch engine serves."""
    g, raw, P, cp = full_bf16
    w = S.make_workload(4, g, B=48)
    cp.set_engine("small")
    try:
        st = check_parity(cp, P, w.H, w.q0, sample_rows(w.B, 8), w.temperature, w.top_k, w.gumbel)
    finally:
        cp.set_engine("auto")
    assert_parity(st)


@pytest.mark.parametrize("fmt", ["bf16", "q8_0"])
@pytest.mark.parametrize("B", [129, 300])
def test_tile_engine_repeated_calls_ragged_chunks(qpk, fmt, B):
    """Row chunks of 128 with a ragged last chunk, called repeatedly: every
    call's sampled frames match the oracle (teacher-forced) and the device
    status stays clear, so no wait between the CTAs that finish a tile
    together ever runs out."""
    import torch
    g = SMALL
    raw = S.make_weights(g, seed=13, gemm_format=fmt, norm_mode="perturbed")
    P = O.Predictor.from_raw(g, raw)
    cp = qpk.CodePredictor(g, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("tile")
        H, q0 = S.toy_inputs(g, B, seed=B)
        rows = sample_rows(B, 12)
        ref = O.predict_frames(P, H[rows], q0[rows], tol=TOL)
        forced = np.zeros((B, g.n_steps), np.int32)
        forced[rows] = ref["codes"]
        tH, tq = torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda()
        tf = torch.from_numpy(forced).cuda()
        for _ in range(5):
            lg = torch.full((B, g.n_steps, g.vocab), float("nan"), device="cuda")
            codes = cp.predict(tH, tq, out_logits=lg, forced=tf)
            torch.cuda.synchronize()
            assert cp.device_status() == 0
            got = lg.cpu().numpy()[rows]
            assert np.isfinite(got).all()
            assert float(np.abs(got - ref["logits"]).max()) <= TOL
            c = codes.cpu().numpy()[rows]
            assert (c[ref["decidable"]] == ref["codes"][ref["decidable"]]).all()
    finally:
        cp.close()
