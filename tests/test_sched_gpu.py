"""State-slot calls (include/qp_sched.h): frames begun into slots and then
advanced one step per call, with the rows of a call at different steps.

A frame run through qp_begin_frames and then steps 2..n_steps, each step fed
the code the oracle chose for the step before (teacher forcing), must give
the oracle's logits at every step and its codes wherever the oracle calls
the decision clear -- whatever order the scheduler visits the frames in and
whichever frames share a call.  Free-running (each step fed the code the
library chose) the calls agree with qp_predict_frames up to each frame's
first near-tie.
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import synthetic as S
from _parity import SMALL, TOL, decided_prefix, run_gpu, sample_rows

pytestmark = pytest.mark.gpu

WIDE_SMALL = dataclasses.replace(SMALL, code_embed_dim=SMALL.talker_hidden)


@pytest.fixture(scope="module")
def qpk():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from codebook_rvq_code_gb300 import build
    build.build()
    import codebook_rvq_code_gb300 as m
    return m


def _handle(qpk, g, seed, max_batch):
    raw = S.make_weights(g, seed=seed, norm_mode="perturbed")
    cp = qpk.CodePredictor(g, max_batch=max_batch)
    cp.load_raw_weights(raw)
    return raw, O.Predictor.from_raw(g, raw), cp


@pytest.fixture(scope="module")
def small(qpk):
    raw, P, cp = _handle(qpk, SMALL, 71, 16)
    yield raw, P, cp
    cp.close()


@pytest.fixture(scope="module")
def wide(qpk):
    raw, P, cp = _handle(qpk, WIDE_SMALL, 72, 16)
    yield raw, P, cp
    cp.close()


class Checker:
    """Accumulates the GPU's logits and codes per (frame, step) against the
    oracle's, teacher-forced to the oracle's codes."""

    def __init__(self, ref, checked=None):
        self.ref = ref
        self.err = 0.0
        self.mismatch = 0
        self.seen = np.zeros(ref["codes"].shape, bool)
        self.checked = None if checked is None else set(int(f) for f in checked)

    def add(self, frames, steps, codes, logits):
        for i, (f, s) in enumerate(zip(frames, steps)):
            j = s - 1
            assert not self.seen[f, j], (f, s)
            self.seen[f, j] = True
            if self.checked is not None and f not in self.checked:
                continue
            self.err = max(self.err, float(np.abs(logits[i] - self.ref["logits"][f, j]).max()))
            if self.ref["decidable"][f, j] and codes[i] != self.ref["codes"][f, j]:
                self.mismatch += 1


def run_schedule(cp, g, H, q0, ref, seed, max_rows=64, checked=None, sampling=None):
    """Frames enter free slots at random ticks; each tick advances a random
    subset of the running frames by one step, in a random row order.  Every
    step's input is ref["codes"]; `checked` limits the comparison to those
    frames.  sampling: None (greedy) or (T, top_k, gumbel [F, n_steps,
    vocab]); each call passes each row's noise for its own step."""
    import torch
    rng = np.random.default_rng(seed)
    F = H.shape[0]
    chk = Checker(ref, checked)
    pending = list(range(F))
    free = list(rng.permutation(cp.max_batch))
    running = {}   # frame -> [slot, next step]
    calls = 0
    while pending or running:
        nb = min(len(pending), len(free), int(rng.integers(0, 5)))
        if nb == 0 and not running:
            nb = min(len(pending), len(free))
        if nb:
            frames = [pending.pop(0) for _ in range(nb)]
            slots = [int(free.pop()) for _ in range(nb)]
            tH = torch.from_numpy(np.ascontiguousarray(H[frames])).cuda()
            tq = torch.from_numpy(q0[frames].astype(np.int32)).cuda()
            lg = torch.empty((nb, g.vocab), dtype=torch.float32, device="cuda")
            smp = None
            if sampling is not None:
                T, k, gum = sampling
                smp = (T, k, torch.from_numpy(np.ascontiguousarray(gum[frames, 0])).cuda())
            q1 = cp.begin_frames(slots, tH, tq, out_logits=lg, sampling=smp)
            chk.add(frames, [1] * nb, q1.cpu().numpy(), lg.cpu().numpy())
            for f, sl in zip(frames, slots):
                running[f] = [sl, 2]
            calls += 1
        ready = list(running)
        if not ready:
            continue
        n = int(rng.integers(1, min(len(ready), max_rows) + 1))
        frames = [ready[i] for i in rng.permutation(len(ready))[:n]]
        slots = [running[f][0] for f in frames]
        steps = [running[f][1] for f in frames]
        cin = torch.from_numpy(np.array([ref["codes"][f, s - 2] for f, s in zip(frames, steps)], np.int32)).cuda()
        lg = torch.empty((n, g.vocab), dtype=torch.float32, device="cuda")
        smp = None
        if sampling is not None:
            T, k, gum = sampling
            smp = (T, k, torch.from_numpy(np.ascontiguousarray(gum[frames, np.array(steps) - 1])).cuda())
        out = cp.step_frames(slots, steps, cin, out_logits=lg, sampling=smp)
        chk.add(frames, steps, out.cpu().numpy(), lg.cpu().numpy())
        calls += 1
        for f in frames:
            running[f][1] += 1
            if running[f][1] > g.n_steps:
                free.append(running.pop(f)[0])
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    assert chk.seen.all()
    return chk, calls


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_ragged_schedule_matches_the_oracle(small, seed):
    raw, P, cp = small
    F = 28
    H, q0 = S.toy_inputs(SMALL, F, seed=500 + seed)
    ref = O.predict_frames(P, H, q0, tol=TOL)
    chk, calls = run_schedule(cp, SMALL, H, q0, ref, seed)
    assert chk.err <= TOL, chk.err
    assert chk.mismatch == 0
    assert ref["decidable"].sum() > 0
    assert calls > F   # the frames were interleaved


@pytest.mark.parametrize("T,k", [(0.9, 50), (0.6, 7), (1.3, 1)])
def test_ragged_schedule_sampling_matches_the_oracle(small, T, k):
    """Gumbel top-k sampling in state-slot calls (qp_begin_frames_ex /
    qp_step_frames_ex): each row decides its own step with that step's noise;
    teacher-forced to the oracle's sampled codes, every clear decision (the
    sampling rule: the winner stays the winner under any change of the logits
    within the tolerance) matches."""
    raw, P, cp = small
    F = 24
    H, q0 = S.toy_inputs(SMALL, F, seed=560 + k)
    gum = S.gumbel_noise((F, SMALL.n_steps, SMALL.vocab), seed=11 + k)
    ref = O.predict_frames(P, H, q0, T, k, gum, tol=TOL)
    chk, calls = run_schedule(cp, SMALL, H, q0, ref, 40 + k, sampling=(T, k, gum))
    assert chk.err <= TOL, chk.err
    assert chk.mismatch == 0
    assert ref["decidable"].sum() > 0
    assert calls > F


def test_sampling_slot_calls_free_running_match_predict(small):
    """Begin, then steps 2..n_steps fed the library's own sampled codes, with
    the noise qp_predict_frames_ex reads for each step, equals one sampled
    qp_predict_frames_ex call up to each frame's first unclear decision."""
    import torch
    raw, P, cp = small
    g = SMALL
    B, T, k = 9, 0.9, 20
    H, q0 = S.toy_inputs(g, B, seed=580)
    gum = S.gumbel_noise((B, g.n_steps, g.vocab), seed=12)
    codes_p, logits_p = run_gpu(cp, H, q0, sampling=(T, k, gum))
    slots = list(range(B))
    codes = np.zeros((B, g.n_steps), np.int32)
    logits = np.zeros((B, g.n_steps, g.vocab), np.float32)
    lg = torch.empty((B, g.vocab), dtype=torch.float32, device="cuda")
    c = cp.begin_frames(slots, torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda(),
                        out_logits=lg, sampling=(T, k, torch.from_numpy(np.ascontiguousarray(gum[:, 0])).cuda()))
    codes[:, 0], logits[:, 0] = c.cpu().numpy(), lg.cpu().numpy()
    for s in range(2, g.n_steps + 1):
        c = cp.step_frames(slots, [s] * B, c, out_logits=lg,
                           sampling=(T, k, torch.from_numpy(np.ascontiguousarray(gum[:, s - 1])).cuda()))
        codes[:, s - 1], logits[:, s - 1] = c.cpu().numpy(), lg.cpu().numpy()
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    ref = O.predict_frames(P, H, q0, T, k, gum, tol=TOL)
    dec = ref["decidable"]
    first = np.where(dec.all(axis=1), g.n_steps, np.argmin(dec, axis=1))
    for b in range(B):   # both runs follow the oracle up to its first unclear decision
        j = first[b]
        np.testing.assert_array_equal(codes[b, :j], codes_p[b, :j])
        assert np.abs(logits[b, :j + 1] - logits_p[b, :j + 1]).max() <= TOL


def test_ragged_schedule_talker_wide_tables(wide):
    raw, P, cp = wide
    F = 20
    H, q0 = S.toy_inputs(WIDE_SMALL, F, seed=520)
    ref = O.predict_frames(P, H, q0, tol=TOL)
    chk, _ = run_schedule(cp, WIDE_SMALL, H, q0, ref, 9)
    assert chk.err <= TOL, chk.err
    assert chk.mismatch == 0


def test_every_step_in_one_call(small):
    """Fourteen rows at steps 2..15 in one call: fourteen step groups, each
    with its own head."""
    import torch
    raw, P, cp = small
    g = SMALL
    F = g.n_steps - 1
    H, q0 = S.toy_inputs(g, F, seed=530)
    ref = O.predict_frames(P, H, q0, tol=TOL)
    chk = Checker(ref)
    slots = list(range(F))
    tH, tq = torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda()
    lg = torch.empty((F, g.vocab), dtype=torch.float32, device="cuda")
    chk.add(range(F), [1] * F, cp.begin_frames(slots, tH, tq, out_logits=lg).cpu().numpy(), lg.cpu().numpy())
    # frame f first catches up to step f + 2 on its own, then all advance together
    for f in range(F):
        for s in range(2, f + 2):
            cin = torch.tensor([ref["codes"][f, s - 2]], dtype=torch.int32, device="cuda")
            l1 = torch.empty((1, g.vocab), dtype=torch.float32, device="cuda")
            chk.add([f], [s], cp.step_frames([f], [s], cin, out_logits=l1).cpu().numpy(), l1.cpu().numpy())
    steps = [f + 2 for f in range(F)]
    order = list(reversed(range(F)))   # rows not in step order
    cin = torch.from_numpy(np.array([ref["codes"][f, steps[f] - 2] for f in order], np.int32)).cuda()
    lg = torch.empty((F, g.vocab), dtype=torch.float32, device="cuda")
    out = cp.step_frames([slots[f] for f in order], [steps[f] for f in order], cin, out_logits=lg)
    chk.add(order, [steps[f] for f in order], out.cpu().numpy(), lg.cpu().numpy())
    assert cp.device_status() == 0
    assert chk.err <= TOL, chk.err
    assert chk.mismatch == 0


@pytest.mark.parametrize("B", [1, 5, 16])
def test_free_running_matches_predict(small, B):
    """Begin, then steps 2..n_steps fed the library's own codes, equals one
    qp_predict_frames call on the same frames (logits without copies)."""
    import torch
    raw, P, cp = small
    g = SMALL
    H, q0 = S.toy_inputs(g, B, seed=540 + B)
    codes_p, logits_p = run_gpu(cp, H, q0)
    slots = list(np.random.default_rng(B).permutation(cp.max_batch)[:B])
    codes = np.zeros((B, g.n_steps), np.int32)
    logits = np.zeros((B, g.n_steps, g.vocab), np.float32)
    lg = torch.empty((B, g.vocab), dtype=torch.float32, device="cuda")
    c = cp.begin_frames(slots, torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda(),
                        out_logits=lg)
    codes[:, 0], logits[:, 0] = c.cpu().numpy(), lg.cpu().numpy()
    for s in range(2, g.n_steps + 1):
        c = cp.step_frames(slots, [s] * B, c, out_logits=lg)
        codes[:, s - 1], logits[:, s - 1] = c.cpu().numpy(), lg.cpu().numpy()
    assert cp.device_status() == 0
    cm, lm = decided_prefix(logits, logits_p)
    np.testing.assert_array_equal(codes[cm], codes_p[cm])
    np.testing.assert_allclose(logits[lm], logits_p[lm], rtol=0, atol=2e-3)


def test_full_size_ragged_calls(qpk):
    """The 1.7B geometry at 32 frames: a ragged schedule teacher-forced to the
    oracle's codes on sampled frames (the oracle computes those frames only;
    the others ride along in the same calls)."""
    import torch
    g = S.Geometry()
    w = S.make_workload(2, g)
    raw = S.make_weights(g, seed=0)
    P = O.Predictor.from_raw(g, raw)
    cp = qpk.CodePredictor(g, max_batch=w.B)
    try:
        cp.load_raw_weights(raw)
        rows = sample_rows(w.B, 4)
        ref_rows = O.predict_frames(P, w.H[rows], w.q0[rows], tol=TOL)
        # the other frames are forced to the codes of a free-running predict call
        codes_p, _ = run_gpu(cp, w.H, w.q0, logits=False)
        forced = codes_p.copy()
        forced[rows] = ref_rows["codes"]
        ref = {"codes": forced, "logits": np.zeros((w.B, g.n_steps, g.vocab), np.float32),
               "decidable": np.zeros((w.B, g.n_steps), bool)}
        ref["logits"][rows] = ref_rows["logits"]
        ref["decidable"][rows] = ref_rows["decidable"]
        chk, calls = run_schedule(cp, g, w.H, w.q0, ref, 4, checked=rows)
        assert chk.err <= TOL, chk.err
        assert chk.mismatch == 0
        assert calls > w.B // 4
    finally:
        cp.close()


def test_state_slot_argument_errors(small, qpk):
    import torch
    raw, P, cp = small
    g = SMALL
    H = torch.zeros((4, g.talker_hidden), device="cuda")
    q0 = torch.zeros(4, dtype=torch.int32, device="cuda")
    c = torch.zeros(4, dtype=torch.int32, device="cuda")
    bad_begin = [
        [0, 1, 1, 2],                 # a slot twice
        [0, 1, 2, cp.max_batch],      # outside the handle's slots
        [0, -1, 2, 3],
    ]
    for slots in bad_begin:
        with pytest.raises(qpk.QpError) as e:
            cp.begin_frames(slots, H, q0)
        assert e.value.code == 1, slots
    for slots, steps in [([0, 1, 2, 3], [2, 2, 1, 2]), ([0, 1, 2, 3], [2, g.n_steps + 1, 2, 2]),
                         ([0, 0, 2, 3], [2, 3, 4, 5])]:
        with pytest.raises(qpk.QpError) as e:
            cp.step_frames(slots, steps, c)
        assert e.value.code == 1, (slots, steps)
    gum = torch.zeros((4, g.vocab), device="cuda")
    for samp in [(0.0, 5, gum), (float("inf"), 5, gum), (0.9, 0, gum), (0.9, g.vocab + 1, gum), (0.9, 5, None)]:
        with pytest.raises(qpk.QpError) as e:
            cp.begin_frames([0, 1, 2, 3], H, q0, sampling=samp)
        assert e.value.code == 1, samp[:2]
        with pytest.raises(qpk.QpError) as e:
            cp.step_frames([0, 1, 2, 3], [2, 2, 2, 2], c, sampling=samp)
        assert e.value.code == 1, samp[:2]
    assert cp.device_status() == 0   # nothing was enqueued


def test_state_slot_bad_codes_latch(small):
    import torch
    raw, P, cp = small
    g = SMALL
    H, q0 = S.toy_inputs(g, 3, seed=560)
    q0 = q0.copy()
    q0[1] = g.q0_vocab + 3
    c = cp.begin_frames([3, 4, 5], torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda())
    assert cp.device_status() == 8
    c = cp.begin_frames([3, 4, 5], torch.from_numpy(H).cuda(), torch.zeros(3, dtype=torch.int32, device="cuda"))
    assert cp.device_status() == 0
    cin = torch.tensor([0, g.vocab, -2], dtype=torch.int32, device="cuda")
    cp.step_frames([3, 4, 5], [2, 2, 2], cin)
    assert cp.device_status() == 8
    assert cp.device_status() == 0


@pytest.mark.parametrize("sampled", [False, True])
def test_state_slots_with_q8_0_weights(qpk, sampled):
    """Q8_0 matrices in state-slot calls (the small-batch engine's hi + lo
    images): a ragged schedule teacher-forced to the oracle's exact d*q
    weights, greedy and sampled."""
    raw = S.make_weights(SMALL, seed=73, gemm_format="q8_0", norm_mode="perturbed")
    P = O.Predictor.from_raw(SMALL, raw)
    cp = qpk.CodePredictor(SMALL, max_batch=16)
    try:
        cp.load_raw_weights(raw)
        F = 18
        H, q0 = S.toy_inputs(SMALL, F, seed=590)
        samp = None
        if sampled:
            samp = (0.9, 40, S.gumbel_noise((F, SMALL.n_steps, SMALL.vocab), seed=13))
        ref = O.predict_frames(P, H, q0, *(samp or (0.0, 0, None)), tol=TOL)
        chk, _ = run_schedule(cp, SMALL, H, q0, ref, 77, sampling=samp)
        assert chk.err <= TOL, chk.err
        assert chk.mismatch == 0
    finally:
        cp.close()


def test_sixty_four_rows_at_mixed_steps(qpk):
    """The largest call: 64 slots, every call holding up to 64 rows spread
    over many steps (uneven step groups), teacher-forced to the oracle."""
    import torch
    g = SMALL
    raw, P, cp = _handle(qpk, g, 74, 64)
    try:
        F = 64
        H, q0 = S.toy_inputs(g, F, seed=570)
        ref = O.predict_frames(P, H, q0, tol=TOL)
        chk = Checker(ref)
        tH, tq = torch.from_numpy(H).cuda(), torch.from_numpy(q0.astype(np.int32)).cuda()
        lg = torch.empty((F, g.vocab), dtype=torch.float32, device="cuda")
        slots = list(range(F))
        chk.add(range(F), [1] * F, cp.begin_frames(slots, tH, tq, out_logits=lg).cpu().numpy(), lg.cpu().numpy())
        nxt = np.full(F, 2)
        tick = 0
        while (nxt <= g.n_steps).any():
            # frame f starts moving at tick f % 9, so the calls hold frames at many steps
            rows = [f for f in range(F) if nxt[f] <= g.n_steps and tick >= f % 9]
            tick += 1
            if not rows:
                continue
            steps = [int(nxt[f]) for f in rows]
            cin = torch.from_numpy(np.array([ref["codes"][f, s - 2] for f, s in zip(rows, steps)], np.int32)).cuda()
            lg = torch.empty((len(rows), g.vocab), dtype=torch.float32, device="cuda")
            out = cp.step_frames([slots[f] for f in rows], steps, cin, out_logits=lg)
            chk.add(rows, steps, out.cpu().numpy(), lg.cpu().numpy())
            nxt[rows] += 1
        assert cp.device_status() == 0
        assert chk.seen.all()
        assert chk.err <= TOL, chk.err
        assert chk.mismatch == 0
    finally:
        cp.close()


def test_misaligned_pointers_are_refused(small, qpk):
    import torch
    raw, P, cp = small
    g = SMALL
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    odd = buf.view(torch.uint8)[1:].data_ptr()   # an int32 array cannot start here
    H = torch.zeros((2, g.talker_hidden), device="cuda")
    lib = cp._lib
    import ctypes
    sl = (ctypes.c_int32 * 2)(0, 1)
    st = (ctypes.c_int32 * 2)(2, 3)
    assert lib.qp_begin_frames(cp._h, 2, sl, H.data_ptr(), odd, buf.data_ptr(), None, None) == 1
    assert lib.qp_begin_frames(cp._h, 2, sl, H.data_ptr(), buf.data_ptr(), odd, None, None) == 1
    assert lib.qp_step_frames(cp._h, 2, sl, st, odd, buf.data_ptr(), None, None) == 1
    assert lib.qp_step_frames(cp._h, 2, sl, st, buf.data_ptr(), buf.data_ptr() + 4 * 8, H.data_ptr() + 4, None) == 1
    assert lib.qp_predict_frames(cp._h, 2, H.data_ptr(), odd, buf.data_ptr(), None, None) == 1
    assert lib.qp_predict_frames(cp._h, 2, H.data_ptr(), buf.data_ptr(), odd, None, None) == 1
    assert cp.device_status() == 0
