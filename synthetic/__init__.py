"""Seeded synthetic weights and inputs for the Qwen3-TTS Code Predictor.

This module only draws numbers: random-init weights in their storage
formats (bf16 bit patterns, raw Q8_0 block streams, f32 vectors), the
per-frame inputs H and q0, and the Gumbel noise a sampling run consumes.
It holds none of the predictor's arithmetic, so both the CPU oracle and the
GPU library can take their inputs from here without sharing any code path.

Tensor names and HF shapes follow the predictor file of
"rightkit-qts 0.2.3 - Qwen3-TTS 1.7B -> QTS GGUF" (sections "Loader contract"
and "Expected verification shapes"); the q0 table is the Talker's
``talker.codec_embd.weight``.  The five workloads are the five batch
configurations the library is measured on (B = 1, 32, 128, 256, 1024).
"""
from __future__ import annotations

from collections import OrderedDict
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional, Tuple

import numpy as np

# storage-type tags (mirrors the names of the C enum qp_dtype)
BF16 = "bf16"
F16 = "f16"
F32 = "f32"
Q8_0 = "q8_0"

Q8_0_BLOCK = 32          # weights per Q8_0 block
Q8_0_BLOCK_BYTES = 34    # one f16 scale + 32 int8 values


@dataclass(frozen=True)
class Geometry:
    """Code Predictor geometry.  Defaults: the 1.7B predictor (1024 hidden,
    5 layers, 16 q-heads / 8 kv-heads of 128, FFN 3072) with 1024-wide code
    embeddings that enter unprojected, a 2048-wide Talker state and 2048-entry
    codebooks."""
    hidden: int = 1024
    layers: int = 5
    n_q_heads: int = 16
    n_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 3072
    vocab: int = 2048
    n_steps: int = 15
    talker_hidden: int = 2048
    code_embed_dim: int = 1024
    q0_vocab: int = 2048
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def q_width(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim


# A toy geometry small enough for brute-force and pure-Python checks.
TOY = Geometry(hidden=64, layers=2, n_q_heads=4, n_kv_heads=2, head_dim=16,
               ffn=96, vocab=37, n_steps=15, talker_hidden=48,
               code_embed_dim=64, q0_vocab=41, rms_eps=1e-6, rope_theta=1e4)


@dataclass
class RawTensor:
    """One weight tensor in its storage format.

    ``data`` is: uint16 bf16 bit patterns shaped ``shape`` (BF16), float32
    (F32), float16 (F16), or uint8 ``[rows, cols/32*34]`` Q8_0 block streams
    (each block: little-endian f16 scale then 32 int8 values, blocks running
    along the input dimension)."""
    name: str
    dtype: str
    shape: Tuple[int, ...]
    data: np.ndarray


def layer_tensor_names(l: int) -> List[str]:
    p = f"code_pred.blk.{l}."
    return [p + s + ".weight" for s in (
        "attn_norm", "attn_q", "attn_k", "attn_v", "attn_output",
        "attn_q_norm", "attn_k_norm", "ffn_norm", "ffn_gate", "ffn_up",
        "ffn_down")]


def tensor_specs(g: Geometry) -> "OrderedDict[str, Tuple[Tuple[int, ...], str]]":
    """Name -> (HF shape [out, in], role) in draw order.

    role is one of 'gemm' (weight matrix), 'bias', 'norm', 'embed', 'head'."""
    s: "OrderedDict[str, Tuple[Tuple[int, ...], str]]" = OrderedDict()
    s["code_pred.small_to_mtp_projection.weight"] = ((g.hidden, g.talker_hidden), "gemm")
    s["code_pred.small_to_mtp_projection.bias"] = ((g.hidden,), "bias")
    s["code_pred.output_norm.weight"] = ((g.hidden,), "norm")
    for l in range(g.layers):
        n = layer_tensor_names(l)
        shapes = [
            ((g.hidden,), "norm"),
            ((g.q_width, g.hidden), "gemm"),
            ((g.kv_width, g.hidden), "gemm"),
            ((g.kv_width, g.hidden), "gemm"),
            ((g.hidden, g.q_width), "gemm"),
            ((g.head_dim,), "norm"),
            ((g.head_dim,), "norm"),
            ((g.hidden,), "norm"),
            ((g.ffn, g.hidden), "gemm"),
            ((g.ffn, g.hidden), "gemm"),
            ((g.hidden, g.ffn), "gemm"),
        ]
        for name, sh in zip(n, shapes):
            s[name] = sh
    for j in range(g.n_steps):
        s[f"code_pred.codec_embd.{j}.weight"] = ((g.vocab, g.code_embed_dim), "embed")
    for j in range(g.n_steps):
        s[f"code_pred.lm_head.{j}.weight"] = ((g.vocab, g.hidden), "head")
    s["talker.codec_embd.weight"] = ((g.q0_vocab, g.talker_hidden), "embed")
    return s


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (storage format only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def pack_q8_0(qs: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Lay out int8 values [rows, cols] and f16 scales [rows, cols/32] as a
    Q8_0 block stream [rows, cols/32*34] (uint8)."""
    rows, cols = qs.shape
    nb = cols // Q8_0_BLOCK
    out = np.empty((rows, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = np.ascontiguousarray(d.astype("<f2")).view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = qs.astype(np.int8).reshape(rows, nb, Q8_0_BLOCK).view(np.uint8)
    return out.reshape(rows, nb * Q8_0_BLOCK_BYTES)


def make_weights(g: Geometry = Geometry(), seed: int = 0, gemm_format: str = BF16,
                 norm_mode: str = "ones", std: float = 0.02,
                 head_format: Optional[str] = None,
                 embed_format: str = BF16) -> "OrderedDict[str, RawTensor]":
    """Random-init predictor weights in storage format.

    * gemm weights: N(0, std) -> bf16 (or f16 with gemm_format == 'f16'), or
      (gemm_format == 'q8_0') int8 values uniform on {-127..127} with one f16
      scale ~ U[1e-4, 2e-3] per 32-block;
    * lm-heads: like gemm weights unless ``head_format`` says otherwise;
    * embeddings: N(0, std) -> bf16, or f16 with embed_format == 'f16' (the
      exporter's layout: f16 embeddings and heads over Q8_0 matrices);
    * bias: N(0, std) f32;  norm vectors: 1.0 ('ones') or 1 + N(0, 0.1)
      ('perturbed', so that a dropped norm-weight multiply is visible), or
      ('wide') the layers' attn_norm and ffn_norm log-uniform on [1, 30] and
      the other norms 1 + N(0, 0.1): large residual-stream operands.
    Everything is drawn from one ``numpy.random.default_rng(seed)`` in the
    order of :func:`tensor_specs`.
    """
    rng = np.random.default_rng(seed)
    head_format = head_format or gemm_format
    out: "OrderedDict[str, RawTensor]" = OrderedDict()
    for name, (shape, role) in tensor_specs(g).items():
        fmt = gemm_format if role == "gemm" else head_format if role == "head" else None
        if role in ("gemm", "head") and fmt == Q8_0:
            rows, cols = shape
            qs = rng.integers(-127, 128, size=(rows, cols), dtype=np.int8)
            d = rng.uniform(1e-4, 2e-3, size=(rows, cols // Q8_0_BLOCK)).astype(np.float16)
            out[name] = RawTensor(name, Q8_0, shape, pack_q8_0(qs, d))
        elif role in ("gemm", "head", "embed"):
            w = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
            f16 = (embed_format if role == "embed" else fmt) == F16
            out[name] = (RawTensor(name, F16, shape, w.astype(np.float16)) if f16
                         else RawTensor(name, BF16, shape, to_bf16_bits(w)))
        elif role == "bias":
            w = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
            out[name] = RawTensor(name, F32, shape, w.astype(np.float32))
        else:  # norm
            if norm_mode == "ones":
                w = np.ones(shape, dtype=np.float32)
            elif norm_mode == "wide" and name.endswith(("attn_norm.weight", "ffn_norm.weight")):
                w = np.exp(rng.uniform(0.0, np.log(30.0), size=shape)).astype(np.float32)
            elif norm_mode in ("perturbed", "wide"):
                w = (1.0 + 0.1 * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)
            else:
                raise ValueError(f"unknown norm_mode {norm_mode!r}")
            out[name] = RawTensor(name, F32, shape, w)
    return out


# ----------------------------------------------------------------------------
# Per-frame inputs for the five batch configurations
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    B: int
    H: np.ndarray                 # float32 [B, talker_hidden]
    q0: np.ndarray                # int32 [B]
    gemm_format: str = BF16
    temperature: float = 0.0      # 0 => greedy
    top_k: int = 0
    gumbel: Optional[np.ndarray] = None   # float32 [B, n_steps, vocab]
    weight_seed: int = 0
    notes: str = ""

    @property
    def greedy(self) -> bool:
        return self.gumbel is None


CONFIG_NAMES = {
    1: "B1_greedy_bf16",
    2: "B32_greedy_bf16_zipf",
    3: "B128_greedy_bf16_ar1",
    4: "B256_topk50_T0.9_bf16",
    5: "B1024_greedy_q8_0",
}


def zipf_codes(rng: np.random.Generator, n: int, vocab: int, s: float) -> np.ndarray:
    """Finite Zipf(s) over ranks 1..vocab by inverse-CDF sampling; code = rank-1."""
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    p = ranks ** (-s)
    cdf = np.cumsum(p / p.sum())
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int32)


def gumbel_noise(shape: Tuple[int, ...], seed: int = 7) -> np.ndarray:
    """Standard Gumbel noise g = -log(-log u), u ~ U(0,1) float32 clamped to
    [1e-20, 1 - 2^-24]."""
    rng = np.random.default_rng(seed)
    u = rng.random(shape, dtype=np.float32)
    u = np.clip(u, np.float32(1e-20), np.float32(1.0 - 2.0 ** -24))
    return (-np.log(-np.log(u))).astype(np.float32)


def make_workload(cfg: int, g: Geometry = Geometry(), B: Optional[int] = None) -> Workload:
    """The inputs of batch configuration ``cfg`` (1..5), seed 100 + cfg.

    ``B`` overrides the batch size (the same recipe at another size)."""
    rng = np.random.default_rng(100 + cfg)
    th, V = g.talker_hidden, g.q0_vocab
    if cfg == 1:
        B = B or 1
        H = rng.standard_normal((B, th), dtype=np.float32)
        q0 = rng.integers(0, V, size=B, dtype=np.int32)
        return Workload(CONFIG_NAMES[1], B, H, q0, notes="H ~ N(0,1); q0 uniform; greedy")
    if cfg == 2:
        B = B or 32
        H = rng.standard_normal((B, th), dtype=np.float32)
        s = rng.uniform(0.5, 2.0, size=(B, 1)).astype(np.float32)
        H = (H * s).astype(np.float32)
        q0 = zipf_codes(rng, B, V, 1.1)
        return Workload(CONFIG_NAMES[2], B, H, q0,
                        notes="H rows N(0,1) x U[0.5,2]; q0 Zipf(1.1); requests 12+12+8; greedy")
    if cfg == 3:
        B = B or 128
        sizes = [13] * 8 + [12] * 2
        if sum(sizes) != B:  # same recipe at another size: requests of ~13 frames
            sizes = [13] * (B // 13) + ([B % 13] if B % 13 else [])
        rows = []
        for n in sizes:
            h = rng.standard_normal(th, dtype=np.float32)
            for t in range(n):
                if t > 0:
                    eps = rng.standard_normal(th, dtype=np.float32)
                    h = (np.float32(0.9) * h + np.float32(np.sqrt(0.19)) * eps).astype(np.float32)
                rows.append(h)
        H = np.stack(rows).astype(np.float32)
        q0 = rng.integers(0, V, size=B, dtype=np.int32)
        return Workload(CONFIG_NAMES[3], B, H, q0,
                        notes="10 requests x ~13 frames, H AR(1) rho=0.9 within a request; greedy")
    if cfg == 4:
        B = B or 256
        H = rng.standard_normal((B, th), dtype=np.float32)
        q0 = rng.integers(0, V, size=B, dtype=np.int32)
        gum = gumbel_noise((B, g.n_steps, g.vocab), seed=7)
        return Workload(CONFIG_NAMES[4], B, H, q0, temperature=0.9, top_k=50, gumbel=gum,
                        notes="H ~ N(0,1); q0 uniform; T=0.9 top-k 50; Gumbel from seed 7")
    if cfg == 5:
        B = B or 1024
        H = rng.standard_normal((B, th), dtype=np.float32)
        q0 = rng.integers(0, V, size=B, dtype=np.int32)
        return Workload(CONFIG_NAMES[5], B, H, q0, gemm_format=Q8_0,
                        notes="H ~ N(0,1); q0 uniform; all GEMM weights Q8_0; greedy")
    raise ValueError(f"unknown config {cfg}")


def workload_weights(w: Workload, g: Geometry = Geometry()) -> "OrderedDict[str, RawTensor]":
    return make_weights(g, seed=w.weight_seed, gemm_format=w.gemm_format)


def toy_inputs(g: Geometry, B: int, seed: int = 5) -> Tuple[np.ndarray, np.ndarray]:
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((B, g.talker_hidden), dtype=np.float32)
    q0 = rng.integers(0, g.q0_vocab, size=B, dtype=np.int32)
    return H, q0
