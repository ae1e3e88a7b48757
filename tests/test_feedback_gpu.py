"""Frame-feedback embeddings (qp_code_embeddings) against the oracle, through
the C ABI: a bf16 -> f32 gather, so bit-exact."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as qpk
    raw = S.make_weights(SMALL, seed=9)
    cp = qpk.CodePredictor(SMALL, max_batch=8)
    cp.load_raw_weights(raw)
    yield qpk, cp, O.Predictor.from_raw(SMALL, raw)
    cp.close()


@pytest.mark.parametrize("B", [1, 5, 300])
def test_code_embeddings_are_bit_exact(setup, B):
    import torch
    qpk, cp, P = setup
    codes = np.random.default_rng(B).integers(0, SMALL.vocab, size=(B, SMALL.n_steps), dtype=np.int32)
    got = cp.code_embeddings(torch.from_numpy(codes).cuda()).cpu().numpy()
    np.testing.assert_array_equal(got, O.code_embeddings(P, codes))
    assert cp.device_status() == 0


def test_code_embeddings_of_predicted_codes(setup):
    """The natural use: embed what qp_predict_frames returned."""
    import torch
    qpk, cp, P = setup
    H, q0 = S.toy_inputs(SMALL, 6, seed=4)
    codes = cp.predict(torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda())
    got = cp.code_embeddings(codes).cpu().numpy()
    np.testing.assert_array_equal(got, O.code_embeddings(P, codes.cpu().numpy()))


def test_out_of_range_codes_latch_bad_token(setup):
    import torch
    qpk, cp, P = setup
    codes = np.zeros((2, SMALL.n_steps), dtype=np.int32)
    codes[1, 3] = SMALL.vocab
    got = cp.code_embeddings(torch.from_numpy(codes).cuda()).cpu().numpy()
    assert cp.device_status() == 8
    np.testing.assert_array_equal(got, O.code_embeddings(P, np.clip(codes, 0, SMALL.vocab - 1)))


def test_empty_and_unloaded(setup):
    import torch
    qpk, cp, P = setup
    out = cp.code_embeddings(torch.zeros((0, SMALL.n_steps), dtype=torch.int32, device="cuda"))
    assert out.shape == (0, SMALL.n_steps, SMALL.hidden)
    fresh = qpk.CodePredictor(SMALL, max_batch=1)
    with pytest.raises(qpk.QpError) as e:
        fresh.code_embeddings(torch.zeros((1, SMALL.n_steps), dtype=torch.int32, device="cuda"))
    assert e.value.code == 2
    fresh.close()
