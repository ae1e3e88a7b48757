"""RVQ codebook normalisation and decode (include/qp_rvq.h) against the
oracle, through the C ABI.  Both are exact in f32: the normalisation is one
IEEE-rounded add and divide per element, the decode adds the stages in the
oracle's order."""
import numpy as np
import pytest

import oracle as O

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


def ema_tables(Q, K, D, seed):
    rng = np.random.default_rng(seed)
    usage = rng.uniform(0.0, 50.0, size=(Q, K)).astype(np.float32)
    usage[:, ::17] = 0.0                                  # unused entries: the literal 1e-7 denominator
    usage[:, 5::29] = rng.uniform(0, 1e-6, size=usage[:, 5::29].shape).astype(np.float32)
    es = (rng.standard_normal((Q, K, D)).astype(np.float32) * usage[:, :, None]).astype(np.float32)
    return es, usage


@pytest.mark.parametrize("Q,K,D", [(16, 2048, 512), (3, 37, 4), (1, 5, 132)])
def test_normalize_is_bit_exact(qpk, Q, K, D):
    import torch
    es, usage = ema_tables(Q, K, D, seed=Q * 7 + D)
    got = qpk.rvq_normalize(torch.from_numpy(es).cuda(), torch.from_numpy(usage).cuda()).cpu().numpy()
    want = np.stack([O.ema_codebook(es[q], usage[q]) for q in range(Q)])
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("Q,K,D,N", [(16, 2048, 512, 1000), (16, 2048, 512, 1), (32, 64, 132, 77),
                                     (1, 9, 4, 5), (7, 100, 260, 333)])
def test_decode_is_bit_exact(qpk, Q, K, D, N):
    import torch
    rng = np.random.default_rng(Q + K + D + N)
    cbs = rng.standard_normal((Q, K, D)).astype(np.float32)
    codes = rng.integers(0, K, size=(N, Q), dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = qpk.rvq_decode(torch.from_numpy(cbs).cuda(), torch.from_numpy(codes).cuda(), status=status).cpu().numpy()
    want = O.rvq_decode(codes, [cbs[q] for q in range(Q)])
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    assert int(status.item()) == 0


def test_decode_of_an_encoding_reconstructs_up_to_the_residual(qpk):
    """x = sum_i C_i[idx_i] + r with the oracle's encoder; the GPU sum is the
    oracle's sum bit for bit."""
    import torch
    rng = np.random.default_rng(11)
    Q, K, D, N = 8, 256, 64, 50
    cbs = [rng.standard_normal((K, D)).astype(np.float32) * (0.5 ** q) for q in range(Q)]
    x = rng.standard_normal((N, D)).astype(np.float32)
    idx, r = O.rvq_encode(x, cbs)
    got = qpk.rvq_decode(torch.from_numpy(np.stack(cbs)).cuda(), torch.from_numpy(idx).cuda()).cpu().numpy()
    np.testing.assert_array_equal(got, O.rvq_decode(idx, cbs))
    np.testing.assert_allclose(got + r, x, rtol=0, atol=1e-5)


def test_out_of_range_codes_are_clamped_and_reported(qpk):
    import torch
    rng = np.random.default_rng(3)
    Q, K, D, N = 4, 10, 8, 6
    cbs = rng.standard_normal((Q, K, D)).astype(np.float32)
    codes = rng.integers(0, K, size=(N, Q), dtype=np.int32)
    codes[2, 1] = K + 3
    codes[4, 3] = -1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = qpk.rvq_decode(torch.from_numpy(cbs).cuda(), torch.from_numpy(codes).cuda(), status=status).cpu().numpy()
    assert int(status.item()) == 8                       # QP_ERR_BAD_TOKEN
    np.testing.assert_array_equal(got, O.rvq_decode(np.clip(codes, 0, K - 1), [cbs[q] for q in range(Q)]))


def test_empty_batch_enqueues_nothing(qpk):
    import torch
    cbs = torch.zeros((2, 3, 4), device="cuda")
    out = qpk.rvq_decode(cbs, torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    assert out.shape == (0, 4)
