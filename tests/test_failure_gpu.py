"""The device-side failure path: a wait that runs out ends the call cleanly.

Every wait inside the frame-loop kernels is bounded.  Here one CTA leaves
one completion count of a GEMM out (include/qp_debug.h, qp_debug_waits), so
the GEMM's consumers wait on a count that never completes; with the wait
limit set to 2 ms the call must latch QP_ERR_TIMEOUT and return within a
fraction of a second (every CTA unwinds; nothing traps), and the next
normal call on the same handle must match the oracle.  The failure is made
by withholding a count, not by any fault.
"""
import time

import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, assert_parity, check_parity

pytestmark = pytest.mark.gpu

QP_ERR_TIMEOUT = 7


@pytest.fixture(scope="module")
def qpk():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m


@pytest.mark.parametrize("engine", ["small", "tile"])
@pytest.mark.parametrize("gemm", [1, 3])   # step 1, layer 0: QKV (attention waits), gate/up (the next GEMM waits)
def test_withheld_count_times_out_and_the_handle_recovers(qpk, engine, gemm):
    import torch
    raw = S.make_weights(SMALL, seed=41, norm_mode="perturbed")
    P = O.Predictor.from_raw(SMALL, raw)
    cp = qpk.CodePredictor(SMALL, max_batch=8)
    try:
        cp.load_raw_weights(raw)
        cp.set_engine(engine)
        H, q0 = S.toy_inputs(SMALL, 5, seed=9)
        tH, tq = torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda()
        cp.predict(tH, tq)                       # a normal call first: one-time set-up is out of the way
        torch.cuda.synchronize()
        assert cp.device_status() == 0
        cp.debug_waits(2000, gemm)
        t0 = time.perf_counter()
        cp.predict(tH, tq)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert cp.device_status() == QP_ERR_TIMEOUT
        assert cp.device_status() == 0           # reading the status clears it
        assert elapsed < 0.5, elapsed            # the 2 ms limit, not the default second
        cp.debug_waits(0, -1)
        assert_parity(check_parity(cp, P, H, q0, np.arange(5)))
    finally:
        cp.close()


def test_debug_waits_rejects_bad_arguments(qpk):
    cp = qpk.CodePredictor(SMALL, max_batch=1)
    try:
        for lim, g in ((-1, -1), (0, -2)):
            with pytest.raises(qpk.QpError) as e:
                cp.debug_waits(lim, g)
            assert e.value.code == 1
    finally:
        cp.close()
