"""GPU-vs-oracle comparison under the three correctness rules.

1. logits within max-abs 3e-2 of the oracle (same bf16 / Q8_0 weights);
2. codes bit-exact at every step the oracle calls decidable (greedy: top-2
   logit gap > 3e-2; sampling: the winner stays the winner under any
   perturbation within 3e-2 / T), with the GPU teacher-forced to the
   oracle's codes so that one near-tie does not derail the rest of a frame;
3. sampling uses the same pre-generated Gumbel noise on both sides.
A free-running GPU pass is also checked: codes agree up to the first
non-decidable step of each frame.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle as O
import synthetic as S

TOL = 3e-2

# A small geometry that keeps head_dim 128 but makes every other size small
# and ragged, so the oracle finishes in a fraction of a second.
SMALL = S.Geometry(hidden=256, layers=2, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=384, vocab=256,
                   n_steps=15, talker_hidden=384, code_embed_dim=256, q0_vocab=300, rms_eps=1e-6,
                   rope_theta=1e6)


def sample_rows(B: int, max_rows: int) -> np.ndarray:
    if B <= max_rows:
        return np.arange(B)
    return np.unique(np.linspace(0, B - 1, max_rows).round().astype(np.int64))


@dataclass
class ParityStats:
    max_abs_logit_err: float
    decidable_steps: int
    total_steps: int
    forced_mismatch: int
    free_prefix_mismatch: int


def run_gpu(cp, H, q0, sampling=None, forced=None, logits=True):
    import torch
    dev = "cuda"
    g = cp.geometry
    B = H.shape[0]
    tH = torch.from_numpy(np.ascontiguousarray(H)).to(dev)
    tq = torch.from_numpy(np.ascontiguousarray(q0.astype(np.int32))).to(dev)
    out_l = torch.empty((B, g.n_steps, g.vocab), dtype=torch.float32, device=dev) if logits else None
    samp = None
    if sampling is not None:
        T, k, gum = sampling
        samp = (T, k, torch.from_numpy(np.ascontiguousarray(gum)).to(dev))
    tf = torch.from_numpy(np.ascontiguousarray(forced.astype(np.int32))).to(dev) if forced is not None else None
    codes = cp.predict(tH, tq, out_logits=out_l, sampling=samp, forced=tf)
    torch.cuda.synchronize()
    st = cp.device_status()
    assert st == 0, f"device status {st}"
    return codes.cpu().numpy(), (out_l.cpu().numpy() if logits else None)


def check_parity(cp, P, H, q0, rows, temperature=0.0, top_k=0, gumbel=None) -> ParityStats:
    g = P.g
    B = H.shape[0]
    sampling = None if gumbel is None else (temperature, top_k, gumbel)
    ref = O.predict_frames(P, H[rows], q0[rows], temperature, top_k,
                           None if gumbel is None else gumbel[rows], tol=TOL)
    forced = np.zeros((B, g.n_steps), np.int32)
    forced[rows] = ref["codes"]
    codes_f, logits_f = run_gpu(cp, H, q0, sampling, forced=forced)
    err = float(np.abs(logits_f[rows] - ref["logits"]).max())
    dec = ref["decidable"]
    mism_forced = int(((codes_f[rows] != ref["codes"]) & dec).sum())
    codes_r, _ = run_gpu(cp, H, q0, sampling, logits=False)
    free_bad = 0
    for i, b in enumerate(rows):
        nd = np.nonzero(~dec[i])[0]
        j = int(nd[0]) if nd.size else g.n_steps
        free_bad += int((codes_r[b, :j] != ref["codes"][i, :j]).sum())
    return ParityStats(err, int(dec.sum()), int(dec.size), mism_forced, free_bad)


def assert_parity(stats: ParityStats):
    assert stats.max_abs_logit_err <= TOL, stats
    assert stats.forced_mismatch == 0, stats
    assert stats.free_prefix_mismatch == 0, stats
    assert stats.decidable_steps > 0, stats


def decided_prefix(*logit_sets, tol: float = TOL):
    """What two free-running calls on the same inputs must agree on.

    A greedy decision whose top-2 gap is within the tolerance may go either
    way between calls (split-K partial sums meet in f32 atomics, in no fixed
    order), and every later step of that frame follows the choice.  So each
    frame agrees up to its first such step, taken over all the given logit
    arrays [B, steps, vocab]: codes before it, logits up to it.  Returns the
    two [B, steps] masks (codes, logits)."""
    clear = np.logical_and.reduce([O.top2_gap(l) > tol for l in logit_sets])
    n = clear.shape[1]
    first = np.where(clear.all(axis=1), n, np.argmin(clear, axis=1))
    steps = np.arange(n)[None, :]
    return steps < first[:, None], steps <= first[:, None]
