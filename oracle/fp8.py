"""FP8 E4M3 KV cache with a per-tensor dynamic scale — oracle.

Sources:
* "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), section 5:
  E4M3 is 1 sign, 4 exponent and 3 mantissa bits; section 6.1: the static
  route fixes every scale to 1.0.
* "大模型量化从0到1（十三）：KV Cache 量化" (CSDN), section 10: ``q = cast_fp8(x/s)``
  and ``x_hat = float(q) * s``; per-tensor granularity (one scale for the whole
  K tensor and another for V).
* "LLM推理加速KV Cache量化压缩实战方案" (yunthe), section "自定义KV Cache量化的实现
  路径": ``scale = max|x| / 448`` with 448 the largest E4M3 value.

E4M3 as used here: exponent bias 7; normal values ``(1 + m/8) * 2^(e-7)`` for
e in 1..15 (except e = 15, m = 7, which is NaN); subnormals ``m/8 * 2^-6``;
largest finite value 448. Encoding rounds to nearest, ties to even; a
magnitude at or above 448 (infinity included) saturates to +-448 (0x7E or
0xFE); every NaN encodes as 0x7F; -0 encodes as 0x80.

Readings: the scale is float32, computed from the fp16 amax as
``fl32(amax / 448)``; an all-zero tensor takes scale 1.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(byte: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    b = np.asarray(byte).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    sub = (m / 8.0) * 2.0 ** -6
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((b & 7) == 7), np.nan, val)


def _round_half_even(x: np.ndarray) -> np.ndarray:
    return np.rint(x)  # numpy rounds halves to even


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """float32 values -> uint8 E4M3 codes (round to nearest even, saturating)."""
    y = np.asarray(y, np.float32).astype(np.float64)
    out = np.zeros(y.shape, np.uint8)
    nan = np.isnan(y)
    sign = np.where(np.signbit(y) & ~nan, 0x80, 0).astype(np.uint8)
    a = np.where(nan, 0.0, np.abs(y))
    sat = a >= E4M3_MAX
    # subnormal grid: multiples of 2^-9 below 2^-6
    sub = a < 2.0 ** -6
    m_sub = _round_half_even(a / 2.0 ** -9)           # 0..8; 8 is the smallest normal (code 0x08)
    # normal grid: exponent from the binade of a, 3 mantissa bits
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # guard against log2 rounding at exact powers of two
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    frac = a / np.exp2(e) - 1.0                        # in [0, 1), exact
    m = _round_half_even(frac * 8.0)                   # 0..8
    e = np.where(m == 8, e + 1, e)
    m = np.where(m == 8, 0, m)
    code_norm = ((e + 7).astype(np.int64) << 3) | m.astype(np.int64)
    code = np.where(sub, m_sub.astype(np.int64), code_norm)
    code = np.where(sat, 0x7E, code)
    out = (code.astype(np.uint8) | sign)
    out = np.where(nan, np.uint8(0x7F), out).astype(np.uint8)
    return out


def amax(x16: np.ndarray) -> np.float32:
    """max |x| over a whole fp16 tensor (exact; NaN if any element is NaN)."""
    return np.float32(np.max(np.abs(x16)))


def dynamic_scale(x16: np.ndarray) -> np.float32:
    """Per-tensor scale ``fl32(amax / 448)``; 1 for an all-zero tensor."""
    a = amax(x16)
    if a == 0:
        return np.float32(1.0)
    return np.float32(a / np.float32(E4M3_MAX))


def quantize(x16: np.ndarray, scale: np.float32) -> np.ndarray:
    """``byte = E4M3(fl32(x / scale))`` elementwise."""
    with np.errstate(divide="ignore", invalid="ignore"):
        y = x16.astype(np.float32) / np.float32(scale)
    return e4m3_encode(y)


def scatter_paged(bytes_bhtd: np.ndarray, block_table: np.ndarray, num_blocks: int, block_size: int) -> np.ndarray:
    """Place token t of sequence b in block ``block_table[b, t // bs]``, row ``t % bs``.

    bytes_bhtd: uint8 ``[B, H, S, D]`` -> pool uint8 ``[num_blocks, H, bs, D]``
    (rows never written stay 0).
    """
    b_, h_, s_, d_ = bytes_bhtd.shape
    pool = np.zeros((num_blocks, h_, block_size, d_), np.uint8)
    for b in range(b_):
        for t0 in range(0, s_, block_size):
            blk = block_table[b, t0 // block_size]
            n = min(block_size, s_ - t0)
            pool[blk, :, :n, :] = bytes_bhtd[b, :, t0:t0 + n, :]
    return pool


def gather_paged(pool: np.ndarray, block_table: np.ndarray, b: int, h: int, seq_len: int) -> np.ndarray:
    """Tokens 0..seq_len-1 of sequence b, kv head h: uint8 ``[seq_len, D]``."""
    bs = pool.shape[2]
    rows = []
    for t0 in range(0, seq_len, bs):
        n = min(bs, seq_len - t0)
        rows.append(pool[block_table[b, t0 // bs], h, :n, :])
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, pool.shape[3]), np.uint8)
