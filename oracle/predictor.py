"""Plain fp32 CPU oracle of the Qwen3-TTS Code Predictor loop.

TEST INFRASTRUCTURE, NOT THE PRODUCT.  Only the test-suite, the smoke check
of ``__graft_entry__`` and the CPU-baseline / reference legs of ``bench.py``
may import or run anything in ``oracle/``.  It shares no code with the CUDA
library; the two meet only in the seeded generators of ``synthetic``.

What it computes, and where the pages say so:

* 15 autoregressive steps per audio frame fill residual codebooks 1..15 after
  the Talker's first code q0 (16 codebooks in all):
  "テキスト音声合成モデルを50ミリ秒未満で応答させる方法", section
  "Qwen3-TTSの最適化方法", item 3 (fixed 15 steps per frame, preallocated KV
  cache, short bounded context); "Qwen3-TTS на Rust", section
  "Архитектура Qwen3-TTS" (16 codebooks, RVQ).
* Inputs are the frame hidden state H and the first code q0; outputs the
  residual codes: "拆解 Qwen3-TTS：OpenVINO 移植过程中的图分离与调度实践",
  section 1 (RVQ diagram: H and q0 feed the short residual loop).
* Geometry and tensors: "rightkit-qts 0.2.3 - Qwen3-TTS 1.7B -> QTS GGUF",
  "Loader contract" (1024 hidden, 5 layers, 16 q / 8 kv heads of 128, FFN
  3072, q width 2048; block tensors attn_norm, attn_q, attn_k, attn_v,
  attn_output, attn_q_norm, attn_k_norm, ffn_norm, ffn_gate, ffn_up,
  ffn_down; small_to_mtp projection with bias; output_norm; 15 codec_embd
  tables and 15 lm_heads) and "Expected verification shapes" (HF [out, in]).
  "No ... RoPE permutation occurs" in the same section: rotate-half RoPE.

Readings taken where the pages are silent:
positions 0 = small_to_mtp(H), 1 = small_to_mtp(E0[q0]), k+1 = E[k-1][q_k]
for k = 1..14 (hidden-wide tables enter unprojected; Talker-wide tables,
2048 x 2048 in the exporter page's shapes, pass through small_to_mtp); RMSNorm x*rsqrt(mean
x^2 + eps)*w; per-head q/k RMSNorm before RoPE; q head h reads kv head
h // (Hq/Hkv); scale 1/sqrt(head_dim); SwiGLU silu(gate)*up; greedy =
lowest index among maxima; sampling = Gumbel-max over the top-k of
logits/T, ordered (value desc, index asc), lowest index on ties.

Everything is float32 (the precision fixed for this oracle).  Weights are
the exact f32 values of their stored form: the bf16 bit patterns, and for
Q8_0 the product d*q of each block's f16 scale and int8 value, which the
GGUF exporter page gives as the weight's value and which is exact in f32.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional

import numpy as np

F32 = np.float32


# ---------------------------------------------------------------------------
# storage formats -> f32
# ---------------------------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> the f32 value it denotes (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def dequant_q8_0(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Q8_0 block stream -> f32 weights.

    Q8_0 ("rightkit-qts 0.2.3", "Upstream differences & verification scope":
    eligible matrices stored as Q8_0 via the GGUF quantiser): blocks of 32
    consecutive weights along the input dimension, each ``{f16 d; int8 q[32]}``,
    value w = d * q.  d*q is exact in f32 (11-bit times 8-bit significand).
    """
    nb = cols // 32
    b = np.ascontiguousarray(blocks).reshape(rows, nb, 34)
    d = np.ascontiguousarray(b[:, :, 0:2]).view("<f2").reshape(rows, nb).astype(np.float32)
    q = np.ascontiguousarray(b[:, :, 2:]).view(np.int8).astype(np.float32)
    return (q * d[:, :, None]).reshape(rows, cols)


def quant_q8_0(w: np.ndarray) -> np.ndarray:
    """f32 [rows, cols] -> Q8_0 block stream, d = max|w| / 127 per block
    (f16), q = round(w / d).  Used only to check the round trip."""
    rows, cols = w.shape
    nb = cols // 32
    wb = w.reshape(rows, nb, 32).astype(np.float32)
    amax = np.abs(wb).max(axis=2)
    d = (amax / F32(127.0)).astype(np.float16)
    dd = d.astype(np.float32)
    inv = np.where(dd > 0, F32(1.0) / np.where(dd > 0, dd, F32(1.0)), F32(0.0))
    q = np.clip(np.rint(wb * inv[:, :, None]), -127, 127).astype(np.int8)
    out = np.empty((rows, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = d.astype("<f2").view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = q.view(np.uint8)
    return out.reshape(rows, nb * 34)


def round_to_f16(w: np.ndarray) -> np.ndarray:
    """f32 -> nearest f16 (ties to even) -> f32."""
    return w.astype(np.float16).astype(np.float32)


def weights_to_f32(raw, q8_0_operand: str = "exact") -> Dict[str, np.ndarray]:
    """Map ``{name: synthetic.RawTensor}`` to ``{name: f32 array}``.

    Q8_0 matrices take their stored value d*q ("rightkit-qts 0.2.3",
    "Upstream differences & verification scope").  ``q8_0_operand='f16'``
    is a diagnostic only: it rounds d*q once to f16, which shows how much
    of a difference a single f16 rounding of the weights accounts for."""
    if q8_0_operand not in ("exact", "f16"):
        raise ValueError(f"q8_0_operand must be 'exact' or 'f16', not {q8_0_operand!r}")
    out = {}
    for name, t in raw.items():
        if t.dtype == "bf16":
            out[name] = bf16_to_f32(t.data).reshape(t.shape)
        elif t.dtype == "q8_0":
            w = dequant_q8_0(t.data, t.shape[0], t.shape[1])
            out[name] = round_to_f16(w) if q8_0_operand == "f16" else w
        elif t.dtype == "f16":
            out[name] = t.data.astype(np.float32).reshape(t.shape)
        elif t.dtype == "f32":
            out[name] = np.asarray(t.data, dtype=np.float32).reshape(t.shape)
        else:
            raise ValueError(f"{name}: unknown storage type {t.dtype}")
    return out


# ---------------------------------------------------------------------------
# the operations of one decoder layer
# ---------------------------------------------------------------------------

def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x * 1/sqrt(mean(x^2) + eps) * w."""
    x = x.astype(F32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=F32)
    return (x * (F32(1.0) / np.sqrt(ms + F32(eps))) * w).astype(F32)


def rope_angles(pos: int, head_dim: int, theta: float):
    """cos/sin of theta_i = pos * theta^(-2i/head_dim), i < head_dim/2.
    The angle is formed in f64 and rounded once to f32."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    ang = pos * theta ** (-2.0 * i / head_dim)
    return np.cos(ang).astype(F32), np.sin(ang).astype(F32)


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE on the last axis (pairs (i, i + head_dim/2)):
    y_i = x_i cos - x_{i+h} sin,  y_{i+h} = x_{i+h} cos + x_i sin."""
    hd = x.shape[-1]
    h = hd // 2
    c, s = rope_angles(pos, hd, theta)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1).astype(F32)


def silu(z: np.ndarray) -> np.ndarray:
    """z / (1 + e^-z); for very negative z, e^-z overflows to inf and the
    quotient is the correct limit 0."""
    with np.errstate(over="ignore"):
        return (z / (F32(1.0) + np.exp(-z))).astype(F32)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_kv_heads: int) -> np.ndarray:
    """Causal GQA attention of one new position over the cached context.

    q [B, Hq, hd]; K, V [B, T, Hkv, hd] hold positions 0..T-1, the last being
    the new position itself, so every key present is at or before the query.
    q head h reads kv head h // (Hq / Hkv).  Softmax in f32, max-subtracted.
    """
    B, Hq, hd = q.shape
    group = Hq // n_kv_heads
    kv_of = np.arange(Hq) // group
    Kh = K[:, :, kv_of, :]                      # [B, T, Hq, hd]
    Vh = V[:, :, kv_of, :]
    s = np.einsum("bhd,bthd->bht", q, Kh).astype(F32) * F32(1.0 / np.sqrt(hd))
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s).astype(F32)
    p = (e / e.sum(axis=-1, keepdims=True, dtype=F32)).astype(F32)
    return np.einsum("bht,bthd->bhd", p, Vh).astype(F32)


@dataclass
class Layer:
    attn_norm: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    q_norm: np.ndarray
    k_norm: np.ndarray
    ffn_norm: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray


class Predictor:
    """f32 weights of the Code Predictor plus its geometry."""

    def __init__(self, g, W: Dict[str, np.ndarray]):
        self.g = g
        self.W = W
        self.layers = []
        for l in range(g.layers):
            p = f"code_pred.blk.{l}."
            self.layers.append(Layer(*[W[p + s + ".weight"] for s in (
                "attn_norm", "attn_q", "attn_k", "attn_v", "attn_output",
                "attn_q_norm", "attn_k_norm", "ffn_norm", "ffn_gate",
                "ffn_up", "ffn_down")]))
        self.w_proj = W["code_pred.small_to_mtp_projection.weight"]
        self.b_proj = W["code_pred.small_to_mtp_projection.bias"]
        self.out_norm = W["code_pred.output_norm.weight"]
        self.embed = [W[f"code_pred.codec_embd.{j}.weight"] for j in range(g.n_steps)]
        self.heads = [W[f"code_pred.lm_head.{j}.weight"] for j in range(g.n_steps)]
        self.e0 = W["talker.codec_embd.weight"]

    @classmethod
    def from_raw(cls, g, raw, q8_0_operand: str = "exact"):
        return cls(g, weights_to_f32(raw, q8_0_operand))

    # -- one decoder layer applied to one new position of every row ---------
    def layer_step(self, l: int, x: np.ndarray, pos: int, cache_k: list, cache_v: list) -> np.ndarray:
        """x [B, d] is the residual stream of position ``pos``; the layer's
        k, v for ``pos`` are appended to cache_k/cache_v (lists over
        positions of [B, Hkv, hd]).  Returns the layer's output stream."""
        g, L = self.g, self.layers[l]
        B = x.shape[0]
        a = rms_norm(x, L.attn_norm, g.rms_eps)
        q = (a @ L.wq.T).reshape(B, g.n_q_heads, g.head_dim)
        k = (a @ L.wk.T).reshape(B, g.n_kv_heads, g.head_dim)
        v = (a @ L.wv.T).reshape(B, g.n_kv_heads, g.head_dim)
        q = rope(rms_norm(q, L.q_norm, g.rms_eps), pos, g.rope_theta)
        k = rope(rms_norm(k, L.k_norm, g.rms_eps), pos, g.rope_theta)
        cache_k.append(k.astype(F32))
        cache_v.append(v.astype(F32))
        K = np.stack(cache_k, axis=1)
        V = np.stack(cache_v, axis=1)
        o = attend(q, K, V, g.n_kv_heads).reshape(B, g.q_width)
        x = (x + o @ L.wo.T).astype(F32)
        m = rms_norm(x, L.ffn_norm, g.rms_eps)
        hmid = silu(m @ L.w_gate.T) * (m @ L.w_up.T)
        return (x + hmid.astype(F32) @ L.w_down.T).astype(F32)

    def project(self, v: np.ndarray) -> np.ndarray:
        """small_to_mtp: Linear talker_hidden -> hidden with bias."""
        return (v.astype(F32) @ self.w_proj.T + self.b_proj).astype(F32)

    def step_input(self, k: int, codes: np.ndarray) -> np.ndarray:
        """The input row of step k >= 2: the code embedding E[k-2][q_{k-1}].

        Tables as wide as the hidden stream enter it unprojected.  Tables as
        wide as the Talker state (2048 x 2048 in "rightkit-qts 0.2.3 --
        Qwen3-TTS 1.7B -> QTS GGUF", section "Expected verification shapes")
        can only enter the 1024-wide stream through small_to_mtp, which the
        same page lists as the predictor's projection: they are projected
        like H and E0[q0] (reading; the page gives the shapes, not the
        wiring)."""
        e = self.embed[k - 2][np.asarray(codes)].astype(F32)
        return self.project(e) if self.g.code_embed_dim != self.g.hidden else e

    def logits(self, step: int, x_last: np.ndarray) -> np.ndarray:
        """lm_head[step-1] applied to the output-normed final stream."""
        y = rms_norm(x_last, self.out_norm, self.g.rms_eps)
        return (y @ self.heads[step - 1].T).astype(F32)


# ---------------------------------------------------------------------------
# decisions
# ---------------------------------------------------------------------------

def greedy_code(logits: np.ndarray) -> np.ndarray:
    """argmax per row, lowest index among equal maxima."""
    return np.argmax(logits, axis=-1).astype(np.int32)


def topk_set(z: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of z, ordered (value desc, index asc)."""
    idx = np.arange(z.shape[0])
    order = np.lexsort((idx, -z))
    return order[:k]


def gumbel_topk_code(logits: np.ndarray, temperature: float, top_k: int, g: np.ndarray) -> int:
    """One row: z = logits / T; S = top-k of z; code = argmax_{i in S} z_i + g_i,
    lowest index among equal maxima."""
    z = (logits / F32(temperature)).astype(F32)
    S = topk_set(z, top_k)
    val = (z[S] + g[S]).astype(F32)
    m = val.max()
    return int(S[val == m].min())


def top2_gap(logits: np.ndarray) -> np.ndarray:
    s = np.sort(logits, axis=-1)
    return (s[..., -1] - s[..., -2]).astype(F32)


def sampling_decidable(logits: np.ndarray, temperature: float, top_k: int, g: np.ndarray,
                       code: int, tol: float) -> bool:
    """Whether any logits within ``tol`` of these give the same sampled code.

    With delta = tol / T: the winner's z must lead the (k+1)-th largest z by
    more than delta (it stays in the top-k), and its z + g must lead, by more
    than delta, that of every other index whose z is within delta of the k-th
    largest or above (every index that could enter the top-k)."""
    z = (logits / F32(temperature)).astype(F32)
    V = z.shape[0]
    order = np.lexsort((np.arange(V), -z))
    delta = tol / temperature
    zk = z[order[top_k - 1]]
    zk1 = z[order[top_k]] if top_k < V else -np.inf
    if not (z[code] - zk1 > delta):
        return False
    cand = np.nonzero(z >= zk - delta)[0]
    cand = cand[cand != code]
    if cand.size == 0:
        return True
    return bool(np.all((z[code] + g[code]) - (z[cand] + g[cand]) > delta))


# ---------------------------------------------------------------------------
# the 15-step loop
# ---------------------------------------------------------------------------

def predict_frames(P: Predictor, H: np.ndarray, q0: np.ndarray,
                   temperature: float = 0.0, top_k: int = 0,
                   gumbel: Optional[np.ndarray] = None,
                   forced: Optional[np.ndarray] = None,
                   tol: float = 3e-2) -> Dict[str, np.ndarray]:
    """Run the Code Predictor over B independent frames.

    H [B, talker_hidden] f32, q0 [B] int.  Greedy when ``gumbel`` is None,
    else Gumbel top-k sampling with the given noise [B, n_steps, vocab].
    ``forced`` [B, n_steps] (teacher forcing): the next step's input uses the
    forced code instead of the decided one; the decided code is still
    reported.  Returns codes [B, n_steps] (q1..q15), logits [B, n_steps, V],
    the top-2 logit gap and a per-step ``decidable`` flag (greedy: gap > tol;
    sampling: :func:`sampling_decidable`).
    """
    g = P.g
    B = H.shape[0]
    n = g.n_steps
    codes = np.zeros((B, n), dtype=np.int32)
    logits = np.zeros((B, n, g.vocab), dtype=np.float32)
    decidable = np.zeros((B, n), dtype=bool)
    caches = [([], []) for _ in range(g.layers)]

    def run_position(x, pos):
        for l in range(g.layers):
            x = P.layer_step(l, x, pos, *caches[l])
        return x

    # step 1 processes positions 0 (H) and 1 (q0); step k >= 2 processes position k
    run_position(P.project(H), 0)
    x = run_position(P.project(P.e0[np.asarray(q0)]), 1)
    for k in range(1, n + 1):
        if k > 1:
            prev = forced[:, k - 2] if forced is not None else codes[:, k - 2]
            x = run_position(P.step_input(k, prev), k)
        lg = P.logits(k, x)
        logits[:, k - 1] = lg
        if gumbel is None:
            codes[:, k - 1] = greedy_code(lg)
            decidable[:, k - 1] = top2_gap(lg) > tol
        else:
            for b in range(B):
                c = gumbel_topk_code(lg[b], temperature, top_k, gumbel[b, k - 1])
                codes[b, k - 1] = c
                decidable[b, k - 1] = sampling_decidable(lg[b], temperature, top_k,
                                                         gumbel[b, k - 1], c, tol)
    return {"codes": codes, "logits": logits, "gap": top2_gap(logits), "decidable": decidable}


# ---------------------------------------------------------------------------
# brute force: the whole prefix, recomputed at every step, no cache
# ---------------------------------------------------------------------------

def forward_sequence(P: Predictor, X: np.ndarray) -> np.ndarray:
    """All positions of a sequence at once, causal mask as a matrix.

    X [B, T, d] -> final residual stream [B, T, d].  Independent of the
    incremental path: no KV cache, scores over all T x T pairs with future
    pairs masked to -inf."""
    g = P.g
    B, T, d = X.shape
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)   # True above the diagonal = future
    x = X.astype(F32)
    for L in P.layers:
        a = rms_norm(x, L.attn_norm, g.rms_eps)
        q = (a @ L.wq.T).reshape(B, T, g.n_q_heads, g.head_dim)
        k = (a @ L.wk.T).reshape(B, T, g.n_kv_heads, g.head_dim)
        v = (a @ L.wv.T).reshape(B, T, g.n_kv_heads, g.head_dim)
        q = rms_norm(q, L.q_norm, g.rms_eps)
        k = rms_norm(k, L.k_norm, g.rms_eps)
        q = np.stack([rope(q[:, t], t, g.rope_theta) for t in range(T)], axis=1)
        k = np.stack([rope(k[:, t], t, g.rope_theta) for t in range(T)], axis=1)
        rep = g.n_q_heads // g.n_kv_heads
        k = np.repeat(k, rep, axis=2)
        v = np.repeat(v, rep, axis=2)
        s = np.einsum("bqhd,bkhd->bhqk", q, k).astype(F32) * F32(1.0 / np.sqrt(g.head_dim))
        s = np.where(mask[None, None], F32(-np.inf), s)
        s = s - s.max(axis=-1, keepdims=True)
        e = np.exp(s)
        p = e / e.sum(axis=-1, keepdims=True)
        o = np.einsum("bhqk,bkhd->bqhd", p, v).reshape(B, T, g.q_width).astype(F32)
        x = (x + o @ L.wo.T).astype(F32)
        m = rms_norm(x, L.ffn_norm, g.rms_eps)
        x = (x + (silu(m @ L.w_gate.T) * (m @ L.w_up.T)) @ L.w_down.T).astype(F32)
    return x


def predict_frames_bruteforce(P: Predictor, H: np.ndarray, q0: np.ndarray,
                              forced: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Greedy loop where step k re-runs :func:`forward_sequence` over the
    whole prefix 0..k (no cache).  For small geometries only."""
    g = P.g
    B = H.shape[0]
    seq = [P.project(H), P.project(P.e0[np.asarray(q0)])]
    codes = np.zeros((B, g.n_steps), dtype=np.int32)
    logits = np.zeros((B, g.n_steps, g.vocab), dtype=np.float32)
    for k in range(1, g.n_steps + 1):
        X = np.stack(seq, axis=1)
        x_last = forward_sequence(P, X)[:, -1]
        lg = P.logits(k, x_last)
        logits[:, k - 1] = lg
        codes[:, k - 1] = greedy_code(lg)
        if k < g.n_steps:
            nxt = forced[:, k - 1] if forced is not None else codes[:, k - 1]
            seq.append(P.step_input(k + 1, nxt))
    return {"codes": codes, "logits": logits}


def code_embeddings(P: Predictor, codes: np.ndarray) -> np.ndarray:
    """Frame-feedback embeddings: out[b, j] = E_j[codes[b, j]] for j < n_steps,
    where codes[b, j] is the frame's code q_{j+1} and E_j the predictor's
    code-embedding table j ("rightkit-qts 0.2.3 -- Qwen3-TTS 1.7B -> QTS GGUF",
    section "Loader contract": code_pred.codec_embd.{0..14}).  The loop reads
    tables 0..n_steps-2 for its own inputs; table n_steps-1 is included here
    (reading: the pages name the tables but not their use outside the loop).
    f32, from the bf16 tables."""
    codes = np.asarray(codes)
    out = np.zeros((codes.shape[0], P.g.n_steps, P.g.code_embed_dim), dtype=F32)
    for j in range(P.g.n_steps):
        out[:, j] = P.embed[j][codes[:, j]]
    return out
