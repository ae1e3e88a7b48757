"""qp_predict_frames_static: the entry point that allocates nothing.

It serves callers that cannot let the library call cudaMalloc for them (their
own allocator holds the GPU's memory, or their audio path forbids allocation
once running): the kernel's scratch sits in a static device array instead.
This checks, through the C ABI, that two calls in a row give what
qp_predict_frames gives on the same handle and inputs, and what the oracle
gives, within the tolerance the parity tests use, on every engine and
weight format the entry point serves, and that sizes beyond the array are
refused.  The file
is collected last so that a failure here never hides another test.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, TOL, decided_prefix

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


def _free_prefix(ref):
    """The oracle's codes and logits that a free-running call must give:
    each frame up to its first near-tie (top-2 gap within the tolerance),
    after which either choice is correct and the frame may follow it."""
    dec = ref["decidable"]
    n = dec.shape[1]
    first = np.where(dec.all(axis=1), n, np.argmin(dec, axis=1))
    steps = np.arange(n)[None, :]
    return steps < first[:, None], steps <= first[:, None]


# Every branch of the entry point: the small-batch engine (bf16, the
# default up to 40 frames), the tile engine's 16-bit kernel (forced) and its
# Q8_0 kernel (every Q8_0 handle), at 1, 5 and 8 frames.
CASES = [("full", 1, "bf16", "auto"), ("full", 8, "bf16", "auto"), ("small", 5, "bf16", "auto"),
         ("full", 1, "bf16", "tile"), ("full", 8, "bf16", "tile"), ("small", 5, "bf16", "tile"),
         ("full", 1, "q8_0", "auto"), ("full", 5, "q8_0", "auto"), ("small", 8, "q8_0", "auto")]


@pytest.mark.parametrize("geo,B,fmt,engine", CASES)
def test_static_entry_matches_the_allocating_entry_and_the_oracle(qpk, geo, B, fmt, engine):
    import torch
    geometry = S.Geometry() if geo == "full" else SMALL
    raw = S.make_weights(geometry, seed=11, norm_mode="perturbed", gemm_format=fmt)
    cp = qpk.CodePredictor(geometry, max_batch=B)
    cp.load_raw_weights(raw)
    cp.set_engine(engine)
    H, q0 = S.toy_inputs(geometry, B, seed=3)
    tH = torch.from_numpy(H).cuda()
    tq = torch.from_numpy(q0.astype(np.int32)).cuda()
    n, V = geometry.n_steps, geometry.vocab
    ref_codes = torch.empty((B, n), dtype=torch.int32, device="cuda")
    ref_logits = torch.empty((B, n, V), dtype=torch.float32, device="cuda")
    lib = cp._lib
    assert lib.qp_predict_frames(cp._h, B, tH.data_ptr(), tq.data_ptr(), ref_codes.data_ptr(),
                                 ref_logits.data_ptr(), None) == 0
    torch.cuda.synchronize()
    ref_l = ref_logits.cpu().numpy()
    ref_c = ref_codes.cpu().numpy()
    orc = O.predict_frames(O.Predictor.from_raw(geometry, raw), H, q0, tol=TOL)
    o_codes, o_logits = _free_prefix(orc)
    for _ in range(2):   # the array keeps the previous call's contents
        codes = torch.full((B, n), -1, dtype=torch.int32, device="cuda")
        logits = torch.full((B, n, V), float("nan"), dtype=torch.float32, device="cuda")
        assert lib.qp_predict_frames_static(cp._h, B, tH.data_ptr(), tq.data_ptr(), codes.data_ptr(),
                                            logits.data_ptr(), None) == 0
        torch.cuda.synchronize()
        assert cp.device_status() == 0
        got_l = logits.cpu().numpy()
        got_c = codes.cpu().numpy()
        assert np.all(np.isfinite(got_l))
        # against the allocating entry on the same handle
        code_mask, logit_mask = decided_prefix(ref_l, got_l)   # near-ties may go either way
        assert np.abs(got_l - ref_l)[logit_mask].max() <= TOL
        np.testing.assert_array_equal(got_c[code_mask], ref_c[code_mask])
        # against the oracle, free-running
        assert np.abs(got_l - orc["logits"])[o_logits].max() <= TOL
        np.testing.assert_array_equal(got_c[o_codes], orc["codes"][o_codes])
    cp.close()


def test_static_entry_refuses_batches_beyond_its_array(qpk):
    import torch
    g = SMALL
    cp = qpk.CodePredictor(g, max_batch=16)
    cp.load_raw_weights(S.make_weights(g, seed=2))
    H = torch.zeros((16, g.talker_hidden), device="cuda")
    q0 = torch.zeros(16, dtype=torch.int32, device="cuda")
    codes = torch.empty((16, g.n_steps), dtype=torch.int32, device="cuda")
    assert cp._lib.qp_predict_frames_static(cp._h, 9, H.data_ptr(), q0.data_ptr(), codes.data_ptr(),
                                            None, None) == 1
    assert cp._lib.qp_predict_frames_static(None, 1, H.data_ptr(), q0.data_ptr(), codes.data_ptr(),
                                            None, None) == 1
    cp.close()
