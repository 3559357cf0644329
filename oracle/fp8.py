"""FP8 KV cache (E4M3, and E5M2) with a per-tensor or per-kv-head scale — oracle.

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

E5M2 (the "大模型量化从0到1（十三）" page, section 18.4: 5 exponent and 2
mantissa bits, more range than E4M3 and less precision): exponent bias 15;
normal values ``(1 + m/4) * 2^(e-15)`` for e in 1..30; subnormals
``m/4 * 2^-14``; e = 31 holds infinity (m = 0) and NaN (m != 0); largest
finite value 57344. Encoding rounds to nearest, ties to even, and saturates:
a magnitude at or above 57344 (infinity included) gives +-57344 (0x7B or
0xFB); every NaN encodes as 0x7F; -0 as 0x80.

Per-head granularity (the same page, section 10.1): one K scale and one V
scale per kv head.

FP8-domain attention (the same page, section 18.7, and the aiinfraguide page's
note on section 6: with FP8 KV and the FlashAttention-3 backend the query is
quantized to FP8 as well, so q.k^T runs on FP8 operands and the query's scale
matters).

Readings: the scale is float32, computed from the fp16 amax as
``fl32(amax / FMAX)`` with FMAX the format's largest finite value (448 for
E4M3, the pages' formula; 57344 for E5M2 by the same rule, which the pages do
not spell out); per kv head the amax is taken over that head's slice (every
batch row, token and channel); an all-zero tensor (or slice) takes scale 1.
For FP8-domain attention the pages give no query scale rule: the query of one
decode step (every batch row, query head and channel) is quantized to E4M3
with the per-tensor rule of the cache, ``fl32(amax_q / 448)``; only q.k^T is
in the FP8 domain (the softmax weights stay in high precision for p.V, which
the pages do not say is quantized).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E5M2_MAX = 57344.0
FORMATS = ("e4m3", "e5m2")


def fmax(fmt: str) -> float:
    return E4M3_MAX if fmt == "e4m3" else E5M2_MAX


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


def e5m2_decode(byte: np.ndarray) -> np.ndarray:
    """uint8 E5M2 codes -> float64 values (inf for 0x7C / 0xFC, NaN for e = 31, m != 0)."""
    b = np.asarray(byte).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 2) & 0x1F
    m = (b & 3).astype(np.float64)
    normal = (1.0 + m / 4.0) * np.exp2((e - 15).astype(np.float64))
    sub = (m / 4.0) * 2.0 ** -14
    val = sign * np.where(e == 0, sub, normal)
    val = np.where((e == 31) & ((b & 3) == 0), sign * np.inf, val)
    return np.where((e == 31) & ((b & 3) != 0), np.nan, val)


def e5m2_encode(y: np.ndarray) -> np.ndarray:
    """float32 values -> uint8 E5M2 codes (round to nearest even, saturating)."""
    with np.errstate(invalid="ignore", divide="ignore"):
        return _e5m2_encode(np.asarray(y, np.float32).astype(np.float64))


def _e5m2_encode(y: np.ndarray) -> np.ndarray:
    nan = np.isnan(y)
    sign = np.where(np.signbit(y) & ~nan, 0x80, 0).astype(np.int64)
    a = np.where(nan, 0.0, np.abs(y))
    sat = a >= E5M2_MAX
    sub = a < 2.0 ** -14
    m_sub = _round_half_even(a / 2.0 ** -16)          # 0..4; 4 is the smallest normal (code 0x04)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(np.exp2(e) > a, e - 1, e)
    e = np.where(np.exp2(e + 1) <= a, e + 1, e)
    frac = a / np.exp2(e) - 1.0                        # in [0, 1), exact
    m = _round_half_even(frac * 4.0)                   # 0..4
    e = np.where(m == 4, e + 1, e)
    m = np.where(m == 4, 0, m)
    code_norm = np.clip((e + 15), 0, 31).astype(np.int64) << 2 | m.astype(np.int64)
    code = np.where(sub, m_sub.astype(np.int64), code_norm)
    code = np.where(sat, 0x7B, code)
    out = (code | sign).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), out).astype(np.uint8)


def decode(byte: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    return e4m3_decode(byte) if fmt == "e4m3" else e5m2_decode(byte)


def encode(y: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    return e4m3_encode(y) if fmt == "e4m3" else e5m2_encode(y)


def amax(x16: np.ndarray) -> np.float32:
    """max |x| over a whole fp16 tensor (exact; NaN if any element is NaN)."""
    return np.float32(np.max(np.abs(x16)))


def _scale_of(a: np.float32, fmt: str) -> np.float32:
    if a == 0:
        return np.float32(1.0)
    return np.float32(np.float32(a) / np.float32(fmax(fmt)))


def dynamic_scale(x16: np.ndarray, fmt: str = "e4m3") -> np.float32:
    """Per-tensor scale ``fl32(amax / FMAX)``; 1 for an all-zero tensor."""
    return _scale_of(amax(x16), fmt)


def dynamic_scale_per_head(x16: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """One scale per kv head of ``x16 [B, H, S, D]``: ``fl32(amax_h / FMAX)``
    with amax_h over that head's slice; 1 for an all-zero slice."""
    return np.array([_scale_of(amax(x16[:, h]), fmt) for h in range(x16.shape[1])], np.float32)


def quantize(x16: np.ndarray, scale, fmt: str = "e4m3") -> np.ndarray:
    """``byte = FP8(fl32(x / scale))`` elementwise. ``scale`` is a scalar or, for
    ``x16 [B, H, S, D]``, one scale per kv head ``[H]``."""
    sc = np.asarray(scale, np.float32)
    if sc.ndim == 1:
        sc = sc.reshape(1, -1, 1, 1)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = x16.astype(np.float32) / sc
    return encode(y, fmt)


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


def quantize_query(q16: np.ndarray):
    """The query of one decode step in E4M3 for FP8-domain attention:
    ``(codes uint8 [B, Hq, D], scale float32)`` with the per-tensor scale
    ``fl32(amax_q / 448)`` (1 for an all-zero query)."""
    scale = dynamic_scale(q16, "e4m3")
    return quantize(q16, scale, "e4m3"), scale


def query_hat(codes: np.ndarray, scale) -> np.ndarray:
    """The query FP8-domain attention uses: ``decode(codes) * scale`` in float64."""
    return e4m3_decode(codes).astype(np.float64) * float(scale)
