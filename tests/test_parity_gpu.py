"""Parity of the CUDA frame loop with the CPU oracle, through the C ABI.

Full-size cases run the five batch configurations at their own B (the
launch configuration the benchmark times) and compare sampled frames that
the oracle recomputes one by one; small-geometry cases compare every frame
at ragged batch sizes, with norm weights perturbed away from 1.
"""
import dataclasses

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
def full_bf16(qpk):
    g = S.Geometry()
    raw = S.make_weights(g, seed=0)
    cp = qpk.CodePredictor(g, max_batch=256)
    cp.load_raw_weights(raw)
    yield g, raw, O.Predictor.from_raw(g, raw), cp
    cp.close()


@pytest.mark.parametrize("cfg,max_rows", [(1, 1), (2, 32), (3, 128), (4, 40)])
def test_full_size_configs_bf16(full_bf16, cfg, max_rows):
    g, raw, P, cp = full_bf16
    w = S.make_workload(cfg, g)
    rows = sample_rows(w.B, max_rows)
    st = check_parity(cp, P, w.H, w.q0, rows, w.temperature, w.top_k, w.gumbel)
    print(cfg, st)
    assert_parity(st)


def test_full_size_config5_q8_0(qpk):
    g = S.Geometry()
    w = S.make_workload(5, g)
    raw = S.workload_weights(w, g)
    P = O.Predictor.from_raw(g, raw)
    cp = qpk.CodePredictor(g, max_batch=w.B)
    cp.load_raw_weights(raw)
    st = check_parity(cp, P, w.H, w.q0, sample_rows(w.B, 24))
    print(5, st)
    cp.close()
    assert_parity(st)


@pytest.fixture(scope="module")
def small(qpk):
    raw = S.make_weights(SMALL, seed=3, norm_mode="perturbed")
    cp = qpk.CodePredictor(SMALL, max_batch=160)
    cp.load_raw_weights(raw)
    yield raw, O.Predictor.from_raw(SMALL, raw), cp
    cp.close()


@pytest.mark.parametrize("B", [1, 2, 3, 33, 130, 160])
def test_small_geometry_greedy_all_rows(small, B):
    raw, P, cp = small
    H, q0 = S.toy_inputs(SMALL, B, seed=B)
    assert_parity(check_parity(cp, P, H, q0, np.arange(B)))


@pytest.mark.parametrize("T,k", [(0.9, 50), (1.3, 1), (0.5, 256), (0.7, 7)])
def test_small_geometry_sampling(small, T, k):
    raw, P, cp = small
    B = 37
    H, q0 = S.toy_inputs(SMALL, B, seed=k)
    gum = S.gumbel_noise((B, SMALL.n_steps, SMALL.vocab), seed=k + 1)
    assert_parity(check_parity(cp, P, H, q0, np.arange(B), T, k, gum))


def test_topk_equal_to_vocab_with_zero_noise_is_greedy(small):
    raw, P, cp = small
    B = 5
    H, q0 = S.toy_inputs(SMALL, B, seed=21)
    zero = np.zeros((B, SMALL.n_steps, SMALL.vocab), np.float32)
    greedy, lg = run_gpu(cp, H, q0)
    sampled, ls = run_gpu(cp, H, q0, sampling=(1.0, SMALL.vocab, zero))
    cm, lm = decided_prefix(lg, ls)
    np.testing.assert_array_equal(greedy[cm], sampled[cm])
    np.testing.assert_allclose(lg[lm], ls[lm], rtol=0, atol=1e-3)


@pytest.mark.parametrize("n_steps", [1, 4])
def test_fewer_steps(qpk, n_steps):
    g = dataclasses.replace(SMALL, n_steps=n_steps)
    raw = S.make_weights(g, seed=4, norm_mode="perturbed")
    cp = qpk.CodePredictor(g, max_batch=9)
    cp.load_raw_weights(raw)
    H, q0 = S.toy_inputs(g, 9, seed=2)
    st = check_parity(cp, O.Predictor.from_raw(g, raw), H, q0, np.arange(9))
    cp.close()
    assert_parity(st)


def test_repeat_calls_agree(small):
    """Split-K partial sums meet in f32 atomics, so two calls may differ in the
    last bits of a logit; they agree far inside the tolerance, and on every
    code, up to each frame's first near-tie."""
    raw, P, cp = small
    H, q0 = S.toy_inputs(SMALL, 17, seed=5)
    a = run_gpu(cp, H, q0)
    b = run_gpu(cp, H, q0)
    cm, lm = decided_prefix(a[1], b[1])
    np.testing.assert_array_equal(a[0][cm], b[0][cm])
    np.testing.assert_allclose(a[1][lm], b[1][lm], rtol=0, atol=1e-3)


def test_host_buffer_entry_matches_device_entry(small):
    raw, P, cp = small
    H, q0 = S.toy_inputs(SMALL, 12, seed=6)
    dev_codes, dev_logits = run_gpu(cp, H, q0)
    host_codes = np.zeros((12, SMALL.n_steps), np.int32)
    cp.predict_host(np.ascontiguousarray(H), q0.astype(np.int32), host_codes)
    cm, _ = decided_prefix(dev_logits)
    np.testing.assert_array_equal(dev_codes[cm], host_codes[cm])


def test_bad_tokens_latch_device_status(small, qpk):
    import torch
    raw, P, cp = small
    H, q0 = S.toy_inputs(SMALL, 4, seed=7)
    q0 = q0.copy()
    q0[2] = SMALL.q0_vocab + 5
    tH = torch.from_numpy(H).cuda()
    cp.predict(tH, torch.from_numpy(q0.astype(np.int32)).cuda())
    assert cp.device_status() == 8
    assert cp.device_status() == 0           # read clears it
    forced = torch.zeros((4, SMALL.n_steps), dtype=torch.int32, device="cuda")
    forced[1, 3] = -1
    cp.predict(tH, torch.from_numpy(S.toy_inputs(SMALL, 4, seed=7)[1].astype(np.int32)).cuda(), forced=forced)
    assert cp.device_status() == 8
    assert cp.device_status() == 0


def test_argument_errors_enqueue_nothing(small, qpk):
    import torch
    raw, P, cp = small
    H = torch.zeros((200, SMALL.talker_hidden), device="cuda")
    q0 = torch.zeros(200, dtype=torch.int32, device="cuda")
    with pytest.raises(qpk.QpError) as e:
        cp.predict(H, q0)                     # B above max_batch
    assert e.value.code == 1
    with pytest.raises(qpk.QpError) as e:
        cp.predict(H[:4], q0[:4], sampling=(0.0, 5, torch.zeros(1, device="cuda")))
    assert e.value.code == 1
    with pytest.raises(qpk.QpError) as e:
        cp.predict(H[:4], q0[:4], sampling=(1.0, SMALL.vocab + 1, torch.zeros(1, device="cuda")))
    assert e.value.code == 1


def test_loader_fails_explicitly(qpk):
    """Missing, unknown, mis-shaped and mixed-format tensors each
    fail the whole load with their own status."""
    import torch
    raw = S.make_weights(SMALL, seed=3)
    cp = qpk.CodePredictor(SMALL, max_batch=2)
    up = {n: (t.dtype, torch.from_numpy(t.data.view(np.uint8).reshape(-1).copy()).cuda(), t.shape)
          for n, t in raw.items()}

    def code_of(d):
        with pytest.raises(qpk.QpError) as e:
            cp.load_weights(d)
        return e.value.code

    d = dict(up); d.pop("code_pred.blk.1.ffn_up.weight")
    assert code_of(d) == 3
    d = dict(up); d["code_pred.blk.9.ffn_up.weight"] = up["code_pred.blk.1.ffn_up.weight"]
    assert code_of(d) == 10
    d = dict(up); n = "code_pred.lm_head.3.weight"; d[n] = (d[n][0], d[n][1], (SMALL.vocab, SMALL.hidden + 128))
    assert code_of(d) == 4
    d = dict(up); n = "code_pred.output_norm.weight"; d[n] = ("bf16", d[n][1], d[n][2])
    assert code_of(d) == 5
    q8 = S.make_weights(SMALL, seed=3, gemm_format="q8_0")
    d = dict(up); n = "code_pred.blk.0.attn_k.weight"
    d[n] = ("q8_0", torch.from_numpy(q8[n].data.reshape(-1).copy()).cuda(), q8[n].shape)
    assert code_of(d) == 5
    with pytest.raises(qpk.QpError) as e:
        cp.predict(torch.zeros((1, SMALL.talker_hidden), device="cuda"), torch.zeros(1, dtype=torch.int32,
                                                                                      device="cuda"))
    assert e.value.code == 2                  # nothing loaded
    cp.load_weights(up)
    cp.close()
