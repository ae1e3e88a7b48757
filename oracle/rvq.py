"""RVQ codebook identities -- TEST INFRASTRUCTURE, NOT THE PRODUCT.

* EMA codebook normalisation: an EMA-trained codebook is stored as a running
  sum of assigned vectors plus a per-entry usage count, and the codebook is
  their ratio, codebook = embedding_sum / (cluster_usage + 1e-7)
  ("Qwen3-TTS на Rust", section "Проблема 1: Формат codebook'ов").
* Residual vector quantisation: stage i quantises the residual left by the
  earlier stages, r_i = x - sum_{j<i} q_j, where q_j is the codebook vector
  stage j picked ("拆解 Qwen3-TTS：OpenVINO 移植过程中的图分离与调度实践",
  section 1, "RVQ 的层级逻辑").  Decoding sums the picked vectors.

Reading: each stage picks the entry nearest (squared L2) to its residual,
lowest index on ties.  Everything is f32.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

F32 = np.float32


def ema_codebook(embedding_sum: np.ndarray, cluster_usage: np.ndarray, eps: float = 1e-7) -> np.ndarray:
    """codebook[c] = embedding_sum[c] / (cluster_usage[c] + eps), element-wise."""
    return (embedding_sum.astype(F32) / (cluster_usage.astype(F32)[:, None] + F32(eps))).astype(F32)


def rvq_encode(x: np.ndarray, codebooks: List[np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    """x [N, D] -> (indices [N, Q], final residual [N, D])."""
    r = x.astype(F32).copy()
    idx = np.zeros((x.shape[0], len(codebooks)), dtype=np.int32)
    for i, C in enumerate(codebooks):
        d2 = ((r[:, None, :] - C[None, :, :]) ** 2).sum(axis=-1)
        pick = np.argmin(d2, axis=1)          # first minimum = lowest index
        idx[:, i] = pick
        r = (r - C[pick]).astype(F32)
    return idx, r


def rvq_decode(idx: np.ndarray, codebooks: List[np.ndarray]) -> np.ndarray:
    """sum_i C_i[idx_i]."""
    out = np.zeros((idx.shape[0], codebooks[0].shape[1]), dtype=F32)
    for i, C in enumerate(codebooks):
        out = (out + C[idx[:, i]]).astype(F32)
    return out
