"""Pins of the CPU oracle against facts outside itself.

Each check below ties one part of the oracle to something it does not
compute: counts and shapes the pages print, closed forms, invariants, a
library routine the special case reduces to, or a brute-force recomputation.
``test_mutants_are_caught`` plants plausible mistakes in copies of the
oracle's functions and asserts that some pin fails for each.
"""
import json
import os

import numpy as np
import pytest

import oracle as O
import synthetic as S
from oracle import predictor as OP

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _toy(seed=1, norm_mode="perturbed"):
    g = S.TOY
    return g, O.Predictor.from_raw(g, S.make_weights(g, seed=seed, norm_mode=norm_mode))


# ---------------------------------------------------------------------------
# pin checks, written against the function under test so mutants can be fed in
# ---------------------------------------------------------------------------

def check_rope(rope_fn) -> bool:
    """RoPE against its complex-number closed form: pairs (x_i, x_{i+h}) as
    x_i + j x_{i+h}, rotated by exp(j p theta^(-2i/hd)); identity at p=0;
    norm preserved; q(m).k(n) depends only on m - n."""
    rng = np.random.default_rng(3)
    hd, theta = 16, 1e4
    x = rng.standard_normal((5, hd)).astype(np.float32)
    ok = True
    for p in (0, 1, 7, 15):
        z = x[:, :hd // 2].astype(np.complex128) + 1j * x[:, hd // 2:].astype(np.complex128)
        ang = p * theta ** (-2.0 * np.arange(hd // 2) / hd)
        zr = z * np.exp(1j * ang)
        want = np.concatenate([zr.real, zr.imag], axis=1)
        got = rope_fn(x, p, theta)
        ok &= np.allclose(got, want, rtol=0, atol=2e-6)
        ok &= np.allclose(np.linalg.norm(got, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)
    ok &= np.array_equal(rope_fn(x, 0, theta), x)
    q, k = x[0], x[1]
    d1 = float(np.dot(rope_fn(q[None], 9, theta)[0], rope_fn(k[None], 4, theta)[0]))
    d2 = float(np.dot(rope_fn(q[None], 6, theta)[0], rope_fn(k[None], 1, theta)[0]))
    ok &= abs(d1 - d2) < 1e-4
    return bool(ok)


def check_attend(attend_fn) -> bool:
    """GQA attention against torch's scaled_dot_product_attention (a library
    routine: scale 1/sqrt(d), kv head h // group), and T=1 gives o = v."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(4)
    B, T, Hq, Hkv, hd = 3, 6, 8, 2, 16
    q = rng.standard_normal((B, Hq, hd)).astype(np.float32)
    K = rng.standard_normal((B, T, Hkv, hd)).astype(np.float32)
    V = rng.standard_normal((B, T, Hkv, hd)).astype(np.float32)
    got = attend_fn(q, K, V, Hkv)
    tq = torch.from_numpy(q)[:, :, None, :]                       # [B, Hq, 1, hd]
    tk = torch.from_numpy(K).permute(0, 2, 1, 3)                   # [B, Hkv, T, hd]
    tv = torch.from_numpy(V).permute(0, 2, 1, 3)
    tk = tk.repeat_interleave(Hq // Hkv, dim=1)
    tv = tv.repeat_interleave(Hq // Hkv, dim=1)
    want = F.scaled_dot_product_attention(tq, tk, tv)[:, :, 0, :].numpy()
    ok = np.allclose(got, want, rtol=1e-5, atol=1e-5)
    one = attend_fn(q, K[:, :1], V[:, :1], Hkv)
    ok &= np.array_equal(one, np.repeat(V[:, 0], Hq // Hkv, axis=1))
    return bool(ok)


def check_rms_norm(rms_fn) -> bool:
    """x=[3,4]: mean square 12.5, so y = x / sqrt(12.5 + eps) * w; w=1 gives
    unit RMS; scale invariance RMSNorm(c x) = RMSNorm(x); w multiplies."""
    x = np.array([[3.0, 4.0]], dtype=np.float32)
    y = rms_fn(x, np.ones(2, np.float32), 0.0)
    ok = np.allclose(y, [[3 / np.sqrt(12.5), 4 / np.sqrt(12.5)]], rtol=1e-6)
    rng = np.random.default_rng(5)
    z = rng.standard_normal((4, 64)).astype(np.float32)
    one = rms_fn(z, np.ones(64, np.float32), 1e-6)
    ok &= np.allclose(np.sqrt((one.astype(np.float64) ** 2).mean(axis=1)), 1.0, rtol=1e-5)
    ok &= np.allclose(rms_fn(z * np.float32(7.5), np.ones(64, np.float32), 1e-6), one, rtol=1e-5, atol=1e-6)
    w = rng.standard_normal(64).astype(np.float32)
    ok &= np.allclose(rms_fn(z, w, 1e-6), one * w, rtol=1e-5, atol=1e-6)
    return bool(ok)


def check_swiglu_order(layer_fn) -> bool:
    """One layer with hand-made weights: attention output zeroed (W_o = 0),
    a constant stream x = 1 so that m = RMSNorm(x) = 1; W_gate = g0/d and
    W_up = 1/d make gate = g0 and up = 1 on every FFN row; W_down = 1/F.
    Then the layer output is 1 + silu(g0) * 1.  g0 = -30 gives ~1; the
    swapped product silu(up) * gate would give 1 - 30 * silu(1)."""
    g = S.Geometry(hidden=8, layers=1, n_q_heads=2, n_kv_heads=1, head_dim=4, ffn=6,
                   vocab=5, n_steps=2, talker_hidden=8, code_embed_dim=8, q0_vocab=5,
                   rms_eps=1e-6, rope_theta=1e4)
    d, F = g.hidden, g.ffn
    W = {}
    for name, (shape, role) in S.tensor_specs(g).items():
        W[name] = np.ones(shape, np.float32) if role == "norm" else np.zeros(shape, np.float32)
    ok = True
    for g0 in (-30.0, 2.0):
        W["code_pred.blk.0.ffn_gate.weight"] = np.full((F, d), g0 / d, np.float32)
        W["code_pred.blk.0.ffn_up.weight"] = np.full((F, d), 1.0 / d, np.float32)
        W["code_pred.blk.0.ffn_down.weight"] = np.full((d, F), 1.0 / F, np.float32)
        P = O.Predictor(g, W)
        x = np.ones((1, d), np.float32)
        out = layer_fn(P, 0, x, 0, [], [])
        want = 1.0 + g0 / (1.0 + np.exp(-g0))
        ok &= np.allclose(out, want, rtol=1e-5, atol=1e-6)
    return bool(ok)


def check_identity_layers(predict_fn) -> bool:
    """With W_o = W_down = 0 every layer is the identity on its stream, so the
    logits at step k are lm_head[k-1] . RMSNorm(input of position k): for k=1
    the projected E0[q0], for k >= 2 the row E[k-2][q_{k-1}]."""
    g = S.TOY
    raw = S.make_weights(g, seed=2, norm_mode="perturbed")
    W = O.weights_to_f32(raw)
    for l in range(g.layers):
        W[f"code_pred.blk.{l}.attn_output.weight"] = np.zeros_like(W[f"code_pred.blk.{l}.attn_output.weight"])
        W[f"code_pred.blk.{l}.ffn_down.weight"] = np.zeros_like(W[f"code_pred.blk.{l}.ffn_down.weight"])
    P = O.Predictor(g, W)
    H, q0 = S.toy_inputs(g, 4, seed=9)
    r = predict_fn(P, H, q0)
    ok = True
    wn = W["code_pred.output_norm.weight"]

    def head(k, x):
        y = x / np.sqrt((x.astype(np.float64) ** 2).mean(axis=1, keepdims=True) + g.rms_eps) * wn
        return y @ W[f"code_pred.lm_head.{k - 1}.weight"].T

    x1 = W["talker.codec_embd.weight"][q0] @ W["code_pred.small_to_mtp_projection.weight"].T \
        + W["code_pred.small_to_mtp_projection.bias"]
    ok &= np.allclose(r["logits"][:, 0], head(1, x1), rtol=1e-4, atol=1e-5)
    for k in range(2, g.n_steps + 1):
        xk = W[f"code_pred.codec_embd.{k - 2}.weight"][r["codes"][:, k - 2]]
        ok &= np.allclose(r["logits"][:, k - 1], head(k, xk), rtol=1e-4, atol=1e-5)
    return bool(ok)


# ---------------------------------------------------------------------------
# the pins
# ---------------------------------------------------------------------------

def test_weight_inventory_matches_the_predictor_file():
    """88 predictor tensors, stored as 36 Q8_0 + 30 F16 + 22 F32 ("rightkit-qts
    0.2.3", output table) under that exporter's rules (vectors F32, embeddings
    and heads F16, matrices Q8_0), plus the Talker's q0 table; the oracle
    reads every one of them."""
    g = S.Geometry()
    specs = S.tensor_specs(g)
    pred = {n: v for n, v in specs.items() if n.startswith("code_pred.")}
    assert len(pred) == 88
    kinds = {"gemm": "Q8_0", "embed": "F16", "head": "F16", "norm": "F32", "bias": "F32"}
    counts = {}
    for n, (shape, role) in pred.items():
        counts[kinds[role]] = counts.get(kinds[role], 0) + 1
    assert counts == {"Q8_0": 36, "F16": 30, "F32": 22}
    shapes = json.load(open(os.path.join(GOLDEN, "hf_shapes.json")))
    for name, shape in shapes["shapes"].items():
        assert tuple(specs[name][0]) == tuple(shape), name

    class Recorder(dict):
        seen = set()

        def __getitem__(self, k):
            self.seen.add(k)
            return dict.__getitem__(self, k)

    t = S.TOY
    W = Recorder(O.weights_to_f32(S.make_weights(t, seed=0)))
    O.Predictor(t, W)
    assert Recorder.seen == set(S.tensor_specs(t))


def test_fifteen_codes_per_frame():
    """15 predicted codebooks per frame, 16 with q0."""
    g, P = _toy()
    H, q0 = S.toy_inputs(g, 2)
    r = O.predict_frames(P, H, q0)
    assert r["codes"].shape == (2, 15) and r["logits"].shape == (2, 15, g.vocab)
    assert 1 + r["codes"].shape[1] == 16
    assert r["codes"].min() >= 0 and r["codes"].max() < g.vocab


def test_cache_equals_full_prefix_recompute():
    """The incremental (KV-cached) loop equals recomputing the whole prefix
    with an explicit causal mask at every step."""
    g, P = _toy()
    H, q0 = S.toy_inputs(g, 3)
    a = O.predict_frames(P, H, q0)
    b = O.predict_frames_bruteforce(P, H, q0)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=1e-5, atol=1e-5)
    forced = np.random.default_rng(0).integers(0, g.vocab, size=(3, 15)).astype(np.int32)
    a = O.predict_frames(P, H, q0, forced=forced)
    b = O.predict_frames_bruteforce(P, H, q0, forced=forced)
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=1e-5, atol=1e-5)


def test_causal_mask_hides_the_future():
    """Changing position j's input leaves every earlier position's output
    bit-identical, and changes position j's own."""
    g, P = _toy()
    rng = np.random.default_rng(6)
    X = rng.standard_normal((2, 9, g.hidden)).astype(np.float32)
    base = O.forward_sequence(P, X)
    for j in (1, 4, 8):
        Y = X.copy()
        Y[:, j] += 1.0
        out = O.forward_sequence(P, Y)
        np.testing.assert_array_equal(out[:, :j], base[:, :j])
        assert not np.allclose(out[:, j], base[:, j])


def test_rope_closed_form():
    assert check_rope(O.rope)


def test_attention_against_library_and_single_position():
    assert check_attend(O.attend)


def test_rms_norm_closed_form():
    assert check_rms_norm(O.rms_norm)


def test_silu_closed_form():
    z = np.array([0.0, 1.0, -1.0, 30.0, -30.0], np.float32)
    want = z / (1.0 + np.exp(-z.astype(np.float64)))
    np.testing.assert_allclose(O.silu(z), want, rtol=1e-6, atol=1e-12)
    assert O.silu(np.float32(1.0)) == pytest.approx(0.7310585786, rel=1e-6)


def test_swiglu_gate_times_up():
    assert check_swiglu_order(O.Predictor.layer_step)


def test_identity_layers_reduce_to_embedding_heads():
    """Pins residual connections, output norm, lm-head index k-1 and code
    embedding index k-2 for the input of step k."""
    assert check_identity_layers(O.predict_frames)


def test_projection_is_affine():
    """small_to_mtp(e_j) = W[:, j] + b; small_to_mtp(0) = b."""
    g, P = _toy()
    e = np.zeros((2, g.talker_hidden), np.float32)
    e[1, 5] = 1.0
    out = P.project(e)
    np.testing.assert_array_equal(out[0], P.b_proj)
    np.testing.assert_allclose(out[1], P.w_proj[:, 5] + P.b_proj, rtol=1e-6)


def test_gqa_with_equal_heads_is_mha():
    """Hkv = Hq: every q head reads its own kv head."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal((2, 4, 8)).astype(np.float32)
    K = rng.standard_normal((2, 3, 4, 8)).astype(np.float32)
    V = rng.standard_normal((2, 3, 4, 8)).astype(np.float32)
    got = O.attend(q, K, V, 4)
    for h in range(4):
        s = np.einsum("bd,btd->bt", q[:, h], K[:, :, h]) / np.sqrt(8)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        np.testing.assert_allclose(got[:, h], np.einsum("bt,btd->bd", p, V[:, :, h]), rtol=1e-5, atol=1e-6)


def test_greedy_takes_lowest_index_on_ties():
    l = np.array([[0.1, 0.7, 0.3, 0.7], [2.0, 2.0, 2.0, 2.0]], np.float32)
    np.testing.assert_array_equal(O.greedy_code(l), [1, 0])


def test_sampling_special_cases_reduce_to_greedy():
    """top-k = 1 is greedy for any noise; top-k = V with zero noise is greedy."""
    rng = np.random.default_rng(10)
    for _ in range(50):
        l = rng.standard_normal(64).astype(np.float32)
        g = rng.gumbel(size=64).astype(np.float32)
        c = int(O.greedy_code(l[None])[0])
        assert O.gumbel_topk_code(l, 0.9, 1, g) == c
        assert O.gumbel_topk_code(l, 0.7, 64, np.zeros(64, np.float32)) == c


def test_topk_set_order_and_boundary_ties():
    z = np.array([1.0, 3.0, 2.0, 3.0, 2.0, 0.5], np.float32)
    np.testing.assert_array_equal(O.topk_set(z, 4), [1, 3, 2, 4])


def test_gumbel_max_matches_softmax_over_topk():
    """Gumbel-max sampling draws index i with probability softmax(z)_i over the
    top-k set and never outside it (chi-square at 0.1% significance)."""
    from scipy import stats
    rng = np.random.default_rng(11)
    l = np.array([1.2, 0.3, -0.5, 2.0, 0.9, -1.0, 0.0, 1.5], np.float32)
    T, k, n = 0.9, 5, 40000
    G = rng.gumbel(size=(n, 8)).astype(np.float32)
    counts = np.zeros(8)
    for i in range(n):
        counts[O.gumbel_topk_code(l, T, k, G[i])] += 1
    S_ = O.topk_set(l / np.float32(T), k)
    outside = np.setdiff1d(np.arange(8), S_)
    assert counts[outside].sum() == 0
    z = l[S_].astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    chi2, pval = stats.chisquare(counts[S_], p * n)
    assert pval > 1e-3, (counts, p * n)


def test_sampling_decidability_rule():
    l = np.zeros(10, np.float32)
    l[3] = 5.0
    g = np.zeros(10, np.float32)
    assert O.sampling_decidable(l, 1.0, 2, g, 3, 3e-2)
    g[0] = 4.999   # a rival within tolerance of winning
    l2 = l.copy()
    l2[0] = 0.0
    assert not O.sampling_decidable(l2, 1.0, 10, g, 3, 3e-2)


def test_teacher_forcing_semantics():
    """Forcing the oracle's own codes changes nothing; forcing other codes
    leaves step 1 unchanged and changes later steps."""
    g, P = _toy()
    H, q0 = S.toy_inputs(g, 3)
    a = O.predict_frames(P, H, q0)
    b = O.predict_frames(P, H, q0, forced=a["codes"])
    np.testing.assert_array_equal(a["logits"], b["logits"])
    other = (a["codes"] + 1) % g.vocab
    c = O.predict_frames(P, H, q0, forced=other)
    np.testing.assert_array_equal(c["logits"][:, 0], a["logits"][:, 0])
    assert not np.allclose(c["logits"][:, 1], a["logits"][:, 1])


def test_ema_codebook_normalisation():
    """codebook = embedding_sum / (cluster_usage + 1e-7): usage 0 divides by
    1e-7 itself; usage 4 gives the mean of 4 vectors; golden hand values."""
    gold = json.load(open(os.path.join(GOLDEN, "ema_codebook.json")))
    es = np.array(gold["embedding_sum"], np.float32)
    cu = np.array(gold["cluster_usage"], np.float32)
    cb = O.ema_codebook(es, cu)
    np.testing.assert_allclose(cb, np.array(gold["codebook"], np.float64), rtol=1e-6)


def test_rvq_residual_identity():
    """x = sum_i C_i[idx_i] + r_final (f32 rounding); with the zero vector in
    every codebook the residual norm never grows."""
    rng = np.random.default_rng(12)
    books = []
    for i in range(16):
        C = (rng.standard_normal((32, 8)) * 0.5 ** i).astype(np.float32)
        C[0] = 0.0
        books.append(C)
    x = rng.standard_normal((50, 8)).astype(np.float32)
    idx, r = O.rvq_encode(x, books)
    np.testing.assert_allclose(O.rvq_decode(idx, books) + r, x, rtol=0, atol=1e-5)
    res = x.copy()
    prev = np.linalg.norm(res, axis=1)
    for i, C in enumerate(books):
        res = res - C[idx[:, i]]
        cur = np.linalg.norm(res, axis=1)
        assert np.all(cur <= prev + 1e-6)
        prev = cur
    np.testing.assert_allclose(res, r, atol=1e-6)


def test_q8_0_dequant_and_round_trip():
    """A hand-packed block decodes to d*q; on-grid weights round-trip exactly."""
    d = np.float16(0.5)
    q = np.arange(-16, 16, dtype=np.int8)
    blk = np.concatenate([np.frombuffer(d.tobytes(), np.uint8), q.view(np.uint8)])[None]
    np.testing.assert_array_equal(O.dequant_q8_0(blk, 1, 32)[0], q.astype(np.float32) * 0.5)
    rng = np.random.default_rng(13)
    dd = rng.uniform(1e-4, 2e-3, size=(4, 2)).astype(np.float16)
    qq = rng.integers(-127, 128, size=(4, 64)).astype(np.int8)
    qq[:, 0] = 127
    qq[:, 32] = -127   # pin |q|max = 127 so the re-derived scale equals dd
    w = qq.astype(np.float32) * np.repeat(dd.astype(np.float32), 32, axis=1)
    back = O.dequant_q8_0(O.quant_q8_0(w), 4, 64)
    np.testing.assert_array_equal(back, w)
    raw = S.pack_q8_0(qq, dd)
    np.testing.assert_array_equal(O.dequant_q8_0(raw, 4, 64), w)


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

def _mutant_rope_sign(x, pos, theta):
    hd = x.shape[-1]; h = hd // 2
    c, s = O.rope_angles(pos, hd, theta)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1).astype(np.float32)


def _mutant_rope_interleaved(x, pos, theta):
    hd = x.shape[-1]
    c, s = O.rope_angles(pos, hd, theta)
    y = x.copy()
    y[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    y[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return y


def _mutant_attend_scale(q, K, V, nkv):
    return OP.attend(q * np.float32(np.sqrt(q.shape[-1])), K, V, nkv)


def _mutant_attend_gqa_modulo(q, K, V, nkv):
    B, Hq, hd = q.shape
    kv_of = np.arange(Hq) % nkv
    s = np.einsum("bhd,bthd->bht", q, K[:, :, kv_of]) / np.sqrt(hd)
    p = np.exp(s - s.max(-1, keepdims=True)); p /= p.sum(-1, keepdims=True)
    return np.einsum("bht,bthd->bhd", p, V[:, :, kv_of]).astype(np.float32)


def _mutant_rms_no_weight(x, w, eps):
    return OP.rms_norm(x, np.ones_like(w), eps)


def _mutant_rms_mean_abs(x, w, eps):
    return (x / (np.mean(np.abs(x), axis=-1, keepdims=True) + eps) * w).astype(np.float32)


def _mutant_layer_swapped_swiglu(self, l, x, pos, ck, cv):
    L = self.layers[l]
    try:
        # swap the roles of gate and up for this call only
        self.layers[l] = OP.Layer(L.attn_norm, L.wq, L.wk, L.wv, L.wo, L.q_norm, L.k_norm,
                                  L.ffn_norm, L.w_up, L.w_gate, L.w_down)
        return O.Predictor.layer_step(self, l, x, pos, ck, cv)
    finally:
        self.layers[l] = L


def _mutant_predict_no_residual(P, H, q0):
    orig = O.Predictor.layer_step

    def step(self, l, x, pos, ck, cv):
        return orig(self, l, x, pos, ck, cv) - x
    O.Predictor.layer_step = step
    try:
        return O.predict_frames(P, H, q0)
    finally:
        O.Predictor.layer_step = orig


def _mutant_predict_head_off_by_one(P, H, q0):
    orig = O.Predictor.logits

    def logits(self, step, x):
        return orig(self, min(step + 1, self.g.n_steps), x)
    O.Predictor.logits = logits
    try:
        return O.predict_frames(P, H, q0)
    finally:
        O.Predictor.logits = orig


def _mutant_predict_no_out_norm(P, H, q0):
    orig = O.Predictor.logits

    def logits(self, step, x):
        return (x @ self.heads[step - 1].T).astype(np.float32)
    O.Predictor.logits = logits
    try:
        return O.predict_frames(P, H, q0)
    finally:
        O.Predictor.logits = orig


@pytest.mark.parametrize("check,mutant", [
    (check_rope, _mutant_rope_sign),
    (check_rope, _mutant_rope_interleaved),
    (check_attend, _mutant_attend_scale),
    (check_attend, _mutant_attend_gqa_modulo),
    (check_rms_norm, _mutant_rms_no_weight),
    (check_rms_norm, _mutant_rms_mean_abs),
    (check_swiglu_order, _mutant_layer_swapped_swiglu),
    (check_identity_layers, _mutant_predict_no_residual),
    (check_identity_layers, _mutant_predict_head_off_by_one),
    (check_identity_layers, _mutant_predict_no_out_norm),
])
def test_mutants_are_caught(check, mutant):
    assert not check(mutant)


def test_mutant_without_cache_append_is_caught():
    """A cache that keeps only the newest position breaks the equality with
    the full-prefix recomputation."""
    g, P = _toy()
    H, q0 = S.toy_inputs(g, 2)
    orig = O.Predictor.layer_step

    def step(self, l, x, pos, ck, cv):
        del ck[:], cv[:]
        return orig(self, l, x, pos, ck, cv)
    O.Predictor.layer_step = step
    try:
        a = O.predict_frames(P, H, q0)
    finally:
        O.Predictor.layer_step = orig
    b = O.predict_frames_bruteforce(P, H, q0, forced=a["codes"])
    assert not np.allclose(a["logits"], b["logits"], rtol=1e-5, atol=1e-5)


def test_q8_0_weight_value_is_exact_d_times_q():
    """By default a Q8_0 weight is d*q itself (the exporter page's value), not
    a rounding of it: the oracle's weights equal the product of the block's
    f16 scale and int8 value formed here in f64, and the f16 diagnostic
    variant is d*q rounded to nearest-even, which numpy's float16
    conversion (a library routine) also gives; values already on the f16
    grid pass unchanged."""
    rng = np.random.default_rng(14)
    qq = rng.integers(-127, 128, size=(3, 64)).astype(np.int8)
    dd = rng.uniform(1e-4, 2e-3, size=(3, 2)).astype(np.float16)
    raw = {"m": S.RawTensor("m", S.Q8_0, (3, 64), S.pack_q8_0(qq, dd))}
    exact = O.weights_to_f32(raw)["m"]
    want = (qq.astype(np.float64).reshape(3, 2, 32) * dd.astype(np.float64)[:, :, None]).reshape(3, 64)
    np.testing.assert_array_equal(exact.astype(np.float64), want)
    got = O.weights_to_f32(raw, "f16")["m"]
    np.testing.assert_array_equal(got, exact.astype(np.float16).astype(np.float32))
    assert np.abs(got - exact).max() <= np.abs(exact).max() * 2.0 ** -11
    on_grid = np.float16([0.5, -0.25, 1.5e-3]).astype(np.float32)
    np.testing.assert_array_equal(O.round_to_f16(on_grid), on_grid)


def test_code_embeddings_take_table_j_for_code_j():
    """Table j answers code j: with column 0 of E_j holding j and column 1 the
    row index c, every output row names its own table and code, so a shifted
    table or a wrong code column fails."""
    import dataclasses
    g = dataclasses.replace(S.TOY, n_steps=5)
    raw = S.make_weights(g, seed=1)
    P = O.Predictor.from_raw(g, raw)
    for j in range(g.n_steps):
        P.embed[j] = np.zeros_like(P.embed[j])
        P.embed[j][:, 0] = j
        P.embed[j][:, 1] = np.arange(P.embed[j].shape[0])
    rng = np.random.default_rng(2)
    codes = rng.integers(0, g.vocab, size=(7, g.n_steps))
    out = O.code_embeddings(P, codes)
    assert out.shape == (7, g.n_steps, g.hidden)
    for j in range(g.n_steps):
        np.testing.assert_array_equal(out[:, j, 0], j)
        np.testing.assert_array_equal(out[:, j, 1], codes[:, j])


# ---------------------------------------------------------------------------
# Talker-wide code embeddings (projected step inputs)
# ---------------------------------------------------------------------------

def _wide_pair(seed=5):
    """Two toy geometries that differ only in how step inputs enter: A has
    Talker-wide (80) code tables that pass through small_to_mtp, B has
    hidden-wide (64) tables that enter unprojected.  A's projection is
    [I | 0] with bias c, and B's tables are A's first 64 columns plus c, so
    every input row is the same in both."""
    import dataclasses
    ga = dataclasses.replace(S.TOY, talker_hidden=80, code_embed_dim=80)
    gb = dataclasses.replace(S.TOY, talker_hidden=80, code_embed_dim=64)
    wa = O.weights_to_f32(S.make_weights(ga, seed=seed, norm_mode="perturbed"))
    rng = np.random.default_rng(seed + 1)
    wp = np.zeros((ga.hidden, ga.talker_hidden), np.float32)
    wp[:, :ga.hidden] = np.eye(ga.hidden, dtype=np.float32)
    c = (0.1 * rng.standard_normal(ga.hidden)).astype(np.float32)
    wa["code_pred.small_to_mtp_projection.weight"] = wp
    wa["code_pred.small_to_mtp_projection.bias"] = c
    wb = dict(wa)
    for j in range(ga.n_steps):
        t = wa[f"code_pred.codec_embd.{j}.weight"]
        wb[f"code_pred.codec_embd.{j}.weight"] = (t[:, :ga.hidden] + c).astype(np.float32)
    return ga, gb, O.Predictor(ga, wa), O.Predictor(gb, wb)


def test_wide_code_tables_are_projected():
    """With the projection [I | 0] + c, Talker-wide tables through
    small_to_mtp give exactly the run of hidden-wide tables holding the
    first columns plus c: the step inputs pass through the projection, its
    bias included, from the right table."""
    ga, gb, PA, PB = _wide_pair()
    H, q0 = S.toy_inputs(ga, 4, seed=9)
    a = O.predict_frames(PA, H, q0)
    b = O.predict_frames(PB, H, q0)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=0, atol=1e-6)
    # and the wide tables do change the result when the projection is not the identity
    rng = np.random.default_rng(11)
    W = dict(PA.W)
    W["code_pred.small_to_mtp_projection.weight"] = (0.1 * rng.standard_normal(
        W["code_pred.small_to_mtp_projection.weight"].shape)).astype(np.float32)
    c = O.predict_frames(O.Predictor(ga, W), H, q0)
    assert np.abs(c["logits"][:, 1:] - a["logits"][:, 1:]).max() > 1e-3


def test_wide_code_tables_cache_equals_full_prefix_recompute():
    import dataclasses
    g = dataclasses.replace(S.TOY, talker_hidden=80, code_embed_dim=80)
    P = O.Predictor.from_raw(g, S.make_weights(g, seed=4, norm_mode="perturbed"))
    H, q0 = S.toy_inputs(g, 3, seed=2)
    a = O.predict_frames(P, H, q0)
    b = O.predict_frames_bruteforce(P, H, q0)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=1e-5, atol=1e-5)
