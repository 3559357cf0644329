"""Single-token decode attention in float64 — oracle.

Source: "大模型量化从0到1（十三）：KV Cache 量化" (CSDN): section 2 gives
``Attention(Q, K, V) = softmax(Q K^T / sqrt(d)) V``; section 3.2 says each
decode step matches the new query against every cached key; section 5 defines
grouped-query attention (several query heads share one K/V head). Section 8
gives how quantization errors enter: ``delta score = q . eps / sqrt(d)`` for
keys and ``o_hat - o = sum_i p_i eps_i`` for values.

Readings: query head ``hq`` uses kv head ``hq // (Hq / Hkv)`` (consecutive
grouping); the scale is the float32 value passed by the caller (by default
``fl32(1/sqrt(D))``), used as a float64 number.
"""
from __future__ import annotations

import numpy as np


def softmax_attend(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, scale: float) -> np.ndarray:
    """One query row against T keys/values, float64.

    q: ``[D]``, k_hat / v_hat: ``[T, D]`` (already dequantized); returns ``[D]``.
    """
    s = (k_hat @ q.astype(np.float64)) * float(scale)
    s = s - s.max()
    p = np.exp(s)
    p /= p.sum()
    return p @ v_hat


def kv_head_of(hq: int, q_heads: int, kv_heads: int) -> int:
    return hq // (q_heads // kv_heads)


def decode_attention(q: np.ndarray, keys_hat, values_hat, kv_heads: int, scale: float, heads=None) -> np.ndarray:
    """Decode attention for every (or the listed) (b, hq).

    q: fp16/float ``[B, Hq, D]``; ``keys_hat(b, h)`` / ``values_hat(b, h)`` return
    float64 ``[T, D]``. Returns float64 ``[B, Hq, D]`` (NaN where not computed).
    """
    b_, hq_, d_ = q.shape
    out = np.full((b_, hq_, d_), np.nan)
    want = heads if heads is not None else [(b, h) for b in range(b_) for h in range(hq_)]
    by_kv = {}
    for b, hq in want:
        by_kv.setdefault((b, kv_head_of(hq, hq_, kv_heads)), []).append(hq)
    for (b, h), hqs in by_kv.items():
        kh, vh = keys_hat(b, h), values_hat(b, h)
        for hq in hqs:
            out[b, hq] = softmax_attend(q[b, hq], kh, vh, scale)
    return out


def default_scale(head_dim: int) -> np.float32:
    return np.float32(1.0) / np.sqrt(np.float32(head_dim))
