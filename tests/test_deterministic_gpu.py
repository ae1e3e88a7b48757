"""Deterministic mode (include/qp.h, qp_set_deterministic).

Repeated calls on identical inputs must give bit-identical logits and codes,
also with other calls in between, for greedy and sampled decisions and for
16-bit and Q8_0 weights; and the mode must still match the oracle under the
usual rules.  (Without the mode, split-K partial sums meet in f32 atomics in
no fixed order and the last bits of the logits vary between calls.)
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


def _calls(cp, w, g, n, other=None):
    import torch
    H, q0 = torch.from_numpy(w.H).cuda(), torch.from_numpy(w.q0).cuda()
    samp = None if w.gumbel is None else (w.temperature, w.top_k, torch.from_numpy(w.gumbel).cuda())
    out = []
    for i in range(n):
        lg = torch.empty((w.B, g.n_steps, g.vocab), dtype=torch.float32, device="cuda")
        codes = cp.predict(H, q0, out_logits=lg, sampling=samp)
        torch.cuda.synchronize()
        assert cp.device_status() == 0
        out.append((codes.cpu().numpy(), lg.cpu().numpy()))
        if other is not None:   # a different call in between
            other()
    return out


@pytest.mark.parametrize("cfg,B,fmt", [(2, 32, "bf16"), (1, 1, "bf16"), (4, 64, "bf16"), (5, 160, "q8_0")])
def test_repeated_calls_are_bit_identical(qpk, cfg, B, fmt):
    import torch
    g = S.Geometry()
    w = S.make_workload(cfg, g, B=B)
    raw = S.make_weights(g, seed=0, gemm_format=fmt)
    cp = qpk.CodePredictor(g, max_batch=B)
    try:
        cp.load_raw_weights(raw)
        cp.set_deterministic(True)
        Ho = torch.randn((B, g.talker_hidden), device="cuda")
        qo = torch.zeros(B, dtype=torch.int32, device="cuda")
        runs = _calls(cp, w, g, 3, other=lambda: cp.predict(Ho, qo))
        for codes, logits in runs[1:]:
            assert np.array_equal(codes, runs[0][0])
            assert np.array_equal(logits.view(np.uint32), runs[0][1].view(np.uint32))
        # and the mode still meets the parity rules against the oracle
        st = check_parity(cp, O.Predictor.from_raw(g, raw), w.H, w.q0, sample_rows(B, 6), w.temperature, w.top_k,
                          w.gumbel)
        print(cfg, B, fmt, st)
        assert_parity(st)
    finally:
        cp.close()


def test_small_geometry_all_rows_deterministic(qpk):
    raw = S.make_weights(SMALL, seed=17, norm_mode="perturbed")
    cp = qpk.CodePredictor(SMALL, max_batch=150)
    try:
        cp.load_raw_weights(raw)
        cp.set_deterministic(True)
        H, q0 = S.toy_inputs(SMALL, 150, seed=4)
        assert_parity(check_parity(cp, O.Predictor.from_raw(SMALL, raw), H, q0, np.arange(150)))
        cp.set_engine("small")   # the small-batch engine has no deterministic schedule
        import torch
        with pytest.raises(qpk.QpError):
            cp.predict(torch.from_numpy(H[:4]).cuda(), torch.from_numpy(q0[:4]).cuda())
    finally:
        cp.close()
