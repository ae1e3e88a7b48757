"""The cluster engine (QP_ENGINE_CLUSTER, include/qp_debug.h) against the
oracle, through the C ABI: the greedy frame loop on 8-CTA clusters, for
geometries with a hidden size of 512 or 1024, an FFN and a
vocabulary that split into 256- and 512-wide jobs, and at most 32 frames;
16-bit or Q8_0 matrices (through their exact f16 hi + lo images), code
tables as wide as the hidden size or as the Talker state (projected at
every step).
"""
import dataclasses
import time

import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import TOL, assert_parity, check_parity, decided_prefix, run_gpu, sample_rows

pytestmark = pytest.mark.gpu

# The smallest geometry the cluster engine serves: two kv groups (two
# attention clusters), two MLP jobs, one head job; the oracle finishes it in
# a fraction of a second.
CL = S.Geometry(hidden=512, layers=2, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=512, vocab=512, n_steps=15,
                talker_hidden=384, code_embed_dim=512, q0_vocab=300, rms_eps=1e-6, rope_theta=1e6)


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
def cl_small(qpk):
    raw = S.make_weights(CL, seed=81, norm_mode="perturbed")
    cp = qpk.CodePredictor(CL, max_batch=32)
    cp.load_raw_weights(raw)
    cp.set_engine("cluster")
    yield raw, O.Predictor.from_raw(CL, raw), cp
    cp.close()


@pytest.mark.parametrize("B", [1, 2, 7, 8, 9, 16, 25, 32])
def test_cluster_small_geometry(cl_small, B):
    raw, P, cp = cl_small
    H, q0 = S.toy_inputs(CL, B, seed=300 + B)
    assert_parity(check_parity(cp, P, H, q0, np.arange(B)))


def test_cluster_agrees_with_the_other_engines(cl_small):
    raw, P, cp = cl_small
    H, q0 = S.toy_inputs(CL, 29, seed=41)
    out = {}
    try:
        for eng in ("cluster", "small", "tile"):
            cp.set_engine(eng)
            out[eng] = run_gpu(cp, H, q0)
    finally:
        cp.set_engine("cluster")
    for eng in ("small", "tile"):
        cm, lm = decided_prefix(out["cluster"][1], out[eng][1])
        np.testing.assert_array_equal(out["cluster"][0][cm], out[eng][0][cm])
        np.testing.assert_allclose(out["cluster"][1][lm], out[eng][1][lm], rtol=0, atol=5e-3)


def test_cluster_repeated_calls(cl_small):
    """Calls on one handle reuse the counters and residual rows (the KV
    cache lives in each CTA's tensor memory for the length of a call)."""
    raw, P, cp = cl_small
    H, q0 = S.toy_inputs(CL, 12, seed=43)
    a = run_gpu(cp, H, q0)
    H2, q2 = S.toy_inputs(CL, 5, seed=44)
    run_gpu(cp, H2, q2)
    b = run_gpu(cp, H, q0)
    cm, lm = decided_prefix(a[1], b[1])
    np.testing.assert_array_equal(a[0][cm], b[0][cm])
    np.testing.assert_allclose(a[1][lm], b[1][lm], rtol=0, atol=5e-3)


@pytest.mark.parametrize("hscale", [1e2, 1e4])
def test_cluster_large_magnitudes(qpk, hscale):
    """H scaled up and norm weights up to x30: operand rows are normalised
    before their f16 conversion (and H slices scaled by a power of two)."""
    raw = S.make_weights(CL, seed=83, norm_mode="wide")
    P = O.Predictor.from_raw(CL, raw)
    cp = qpk.CodePredictor(CL, max_batch=8)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(CL, 8, seed=45)
        assert_parity(check_parity(cp, P, (H * hscale).astype(np.float32), q0, np.arange(8)))
    finally:
        cp.close()


@pytest.mark.parametrize("B", [1, 32])
def test_cluster_full_geometry(qpk, B):
    """The 1.7B predictor's geometry (8 attention clusters, 12 MLP jobs, 4
    head jobs), sampled frames against the oracle."""
    g = S.Geometry()
    raw = S.make_weights(g, seed=85, norm_mode="perturbed")
    P = O.Predictor.from_raw(g, raw)
    cp = qpk.CodePredictor(g, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(g, B, seed=46 + B)
        assert_parity(check_parity(cp, P, H, q0, sample_rows(B, 4)))
    finally:
        cp.close()


def test_cluster_refuses_what_it_cannot_serve(qpk, cl_small):
    import torch
    raw, P, cp = cl_small
    H = torch.zeros((33, CL.talker_hidden), device="cuda")
    q0 = torch.zeros(33, dtype=torch.int32, device="cuda")
    big = qpk.CodePredictor(CL, max_batch=40)
    try:
        big.load_raw_weights(raw)
        big.set_engine("cluster")
        with pytest.raises(qpk.QpError) as e:
            big.predict(H, q0)                     # more than 32 frames
        assert e.value.code == 1
        big.predict(H[:32], q0[:32])               # 32 are served
        torch.cuda.synchronize()
        assert big.device_status() == 0
        gum = torch.zeros((2, CL.n_steps, CL.vocab), device="cuda")
        with pytest.raises(qpk.QpError):
            big.predict(H[:2], q0[:2], sampling=(0.8, 10, gum))   # sampling
    finally:
        big.close()
    small_geo = dataclasses.replace(CL, hidden=256, code_embed_dim=256)   # hidden below 512
    sm = qpk.CodePredictor(small_geo, max_batch=4)
    try:
        sm.load_raw_weights(S.make_weights(small_geo, seed=88))
        sm.set_engine("cluster")
        with pytest.raises(qpk.QpError):
            sm.predict(torch.zeros((2, small_geo.talker_hidden), device="cuda"), q0[:2])
    finally:
        sm.close()


@pytest.mark.parametrize("B", [3, 25])
def test_cluster_seven_layers_fill_tensor_memory(qpk, B):
    """Seven layers use all 512 tensor-memory columns (the 64-column
    accumulator, then 64 columns of KV cache per layer): served and checked
    against the oracle with the per-CTA and the shared-load operand builds;
    an eighth layer is refused, and the automatic choice serves it on
    another engine."""
    import torch
    g7 = dataclasses.replace(CL, layers=7)
    raw = S.make_weights(g7, seed=93, norm_mode="perturbed")
    cp = qpk.CodePredictor(g7, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(g7, B, seed=95 + B)
        assert_parity(check_parity(cp, O.Predictor.from_raw(g7, raw), H, q0, sample_rows(B, 4)))
    finally:
        cp.close()
    g8 = dataclasses.replace(CL, layers=8)
    raw8 = S.make_weights(g8, seed=94, norm_mode="perturbed")
    cp = qpk.CodePredictor(g8, max_batch=B)
    try:
        cp.load_raw_weights(raw8)
        H, q0 = S.toy_inputs(g8, B, seed=97)
        tH, tq = torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda()
        cp.set_engine("cluster")
        with pytest.raises(qpk.QpError) as e:
            cp.predict(tH, tq)
        assert e.value.code == 1
        cp.set_engine("auto")
        assert_parity(check_parity(cp, O.Predictor.from_raw(g8, raw8), H, q0, sample_rows(B, 2)))
    finally:
        cp.close()


def test_cluster_bad_first_code_is_reported(cl_small):
    import torch
    raw, P, cp = cl_small
    H = torch.zeros((3, CL.talker_hidden), device="cuda")
    q0 = torch.tensor([0, CL.q0_vocab, 5], dtype=torch.int32, device="cuda")
    cp.predict(H, q0)
    torch.cuda.synchronize()
    assert cp.device_status() == 8    # QP_ERR_BAD_TOKEN, latched (reading clears it)
    H2, q2 = S.toy_inputs(CL, 4, seed=47)
    assert_parity(check_parity(cp, P, H2, q2, np.arange(4)))


def test_cluster_withheld_count_times_out_and_the_handle_recovers(qpk):
    """A count that never arrives (CTA 0's attention count at step 1, layer
    0): the MLP jobs' waits run out after the 2 ms limit, every cluster
    unwinds, and the next call on the handle is correct."""
    import torch
    raw = S.make_weights(CL, seed=89, norm_mode="perturbed")
    P = O.Predictor.from_raw(CL, raw)
    cp = qpk.CodePredictor(CL, max_batch=8)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(CL, 5, seed=48)
        tH, tq = torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda()
        cp.predict(tH, tq)
        torch.cuda.synchronize()
        assert cp.device_status() == 0
        cp.debug_waits(2000, 0)
        t0 = time.perf_counter()
        cp.predict(tH, tq)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert cp.device_status() == 7           # QP_ERR_TIMEOUT
        assert elapsed < 0.5, elapsed
        cp.debug_waits(0, -1)
        assert_parity(check_parity(cp, P, H, q0, np.arange(5)))
    finally:
        cp.close()


@pytest.mark.parametrize("B", [1, 9, 32])
def test_cluster_q8_0(qpk, B):
    """Q8_0 matrices through their f16 hi + lo images (two slices per unit)
    against the oracle's exact d*q weights."""
    raw = S.make_weights(CL, seed=90 + B, gemm_format="q8_0", norm_mode="perturbed")
    P = O.Predictor.from_raw(CL, raw)
    cp = qpk.CodePredictor(CL, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(CL, B, seed=49 + B)
        assert_parity(check_parity(cp, P, H, q0, np.arange(B)))
    finally:
        cp.close()


CL_WIDE = dataclasses.replace(CL, code_embed_dim=CL.talker_hidden)


@pytest.mark.parametrize("B,fmt", [(1, "bf16"), (17, "bf16"), (3, "q8_0"), (32, "q8_0")])
def test_cluster_wide_tables(qpk, B, fmt):
    """Talker-wide code tables: each step's input row is projected by a GEMM
    spread over all CTAs; with Q8_0 the exporter's layout (f16 heads and
    tables over Q8_0 matrices)."""
    kw = {"gemm_format": fmt}
    if fmt == "q8_0":
        kw.update(head_format="f16", embed_format="f16")
    raw = S.make_weights(CL_WIDE, seed=94 + B, norm_mode="perturbed", **kw)
    P = O.Predictor.from_raw(CL_WIDE, raw)
    cp = qpk.CodePredictor(CL_WIDE, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(CL_WIDE, B, seed=53 + B)
        assert_parity(check_parity(cp, P, H, q0, np.arange(B)))
    finally:
        cp.close()


@pytest.mark.parametrize("B", [1, 32])
def test_cluster_exporter_layout_full_geometry(qpk, B):
    """The exporter's real-model layout at the 1.7B geometry (2048-wide code
    tables, Q8_0 matrices, f16 heads and tables), sampled frames against the
    oracle."""
    g = dataclasses.replace(S.Geometry(), code_embed_dim=S.Geometry().talker_hidden)
    raw = S.make_weights(g, seed=97, gemm_format="q8_0", head_format="f16", embed_format="f16",
                         norm_mode="perturbed")
    P = O.Predictor.from_raw(g, raw)
    cp = qpk.CodePredictor(g, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine("cluster")
        H, q0 = S.toy_inputs(g, B, seed=58 + B)
        assert_parity(check_parity(cp, P, H, q0, sample_rows(B, 3)))
    finally:
        cp.close()


def test_cluster_bad_forced_code_is_reported(cl_small):
    """A forced code outside [0, vocab) latches QP_ERR_BAD_TOKEN and is
    clamped; the call still finishes."""
    import torch
    raw, P, cp = cl_small
    H, q0 = S.toy_inputs(CL, 4, seed=61)
    forced = np.zeros((4, CL.n_steps), np.int32)
    forced[2, 5] = CL.vocab + 3
    cp.predict(torch.from_numpy(H).cuda(), torch.from_numpy(q0).cuda(),
               forced=torch.from_numpy(forced).cuda())
    torch.cuda.synchronize()
    assert cp.device_status() == 8    # QP_ERR_BAD_TOKEN
    assert cp.device_status() == 0


def test_cluster_deterministic_mode_goes_to_the_tile_engine(qpk, cl_small):
    """The deterministic schedule is the tile engine's: forcing the cluster
    engine with it is refused, AUTO serves it."""
    import torch
    raw, P, cp = cl_small
    H, q0 = S.toy_inputs(CL, 3, seed=62)
    tH, tq = torch.from_numpy(H).cuda(), torch.from_numpy(q0).cuda()
    cp.set_deterministic(True)
    try:
        with pytest.raises(qpk.QpError) as e:
            cp.predict(tH, tq)
        assert e.value.code == 1
        cp.set_engine("auto")
        a = cp.predict(tH, tq).cpu().numpy()
        b = cp.predict(tH, tq).cpu().numpy()
        np.testing.assert_array_equal(a, b)
    finally:
        cp.set_deterministic(False)
        cp.set_engine("cluster")


def test_cluster_stress_random_batches(cl_small):
    """Forty calls back to back with random batch sizes (both kernel
    instantiations), teacher-forced to the tile engine's codes: every call's
    logits match the tile engine's on the same inputs, so no buffer, counter
    or cluster barrier of one call leaks into the next."""
    import torch
    raw, P, cp = cl_small
    rng = np.random.default_rng(7)
    for it in range(40):
        B = int(rng.integers(1, 33))
        H, q0 = S.toy_inputs(CL, B, seed=1000 + it)
        try:
            cp.set_engine("tile")
            codes_t, logits_t = run_gpu(cp, H, q0)
            cp.set_engine("cluster")
            codes_c, logits_c = run_gpu(cp, H, q0, forced=codes_t)
        finally:
            cp.set_engine("cluster")
        err = float(np.abs(logits_c - logits_t).max())
        assert err <= 5e-3, (it, B, err)
