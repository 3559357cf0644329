"""NVFP4 KV cache (4-bit E2M1 values, E4M3 block scales, fp32 tensor scale) — oracle.

Source: "大模型量化从0到1（十三）：KV Cache 量化" (CSDN), section 21.2 (NVFP4 KV
Cache: a more aggressive 4-bit floating-point KV path in TensorRT-LLM, its
scales produced offline by a calibration tool, for Blackwell-class GPUs) and
section 21.3 (about 1/4 of the BF16 bytes; more calibration-sensitive than
FP8). The pages give no bit format, so this module follows NVIDIA's public
NVFP4 definition (the format of Blackwell's block-scaled tensor cores), with
the pages' per-tensor amax rule for the tensor scale:

* element: FP4 E2M1 — 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit;
  code bits ``s e1 e0 m``; exponent field 0 is subnormal, ``m * 0.5``;
  otherwise ``(1 + m/2) * 2^(E-1)``: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
  Encoding rounds to nearest, ties to the even code, and saturates: a
  magnitude above 6 gives +-6. There is no infinity or NaN: inputs must be
  finite (reading, as for the KIVI path).
* block: 16 consecutive elements of one token along head_dim (channels
  16j .. 16j + 15) share one scale stored as an E4M3 byte (``oracle.fp8``).
* tensor: one float32 scale for the whole K (or V) tensor of the layer.

Readings (the scale rule; the pages leave it to the calibration tool):
* tensor scale ``s_t = fl32(amax / 2688)`` with amax = max |x| over the
  tensor and 2688 = 448 * 6, the largest magnitude a block scale times an
  element can represent (the pages' ``amax / FMAX`` rule with the format's
  FMAX); 1 for an all-zero tensor. A static (calibrated) ``s_t`` is taken as
  given.
* block scale byte ``b = E4M3(fl32(fl32(amax_b / 6) / s_t))`` with amax_b =
  max |x| over the 16 elements: the block's largest element lands on the top
  E2M1 value 6; decoded block scale ``S_b = e4m3(b)``.
* element code ``E2M1(fl32(x / fl32(S_b * s_t)))``; every code of a block is
  0 when ``S_b = 0``.
* dequantized value ``e2m1(code) * S_b * s_t`` (exact in float64).
"""
from __future__ import annotations

import numpy as np

from oracle import fp8

BLOCK = 16
E2M1_MAX = 6.0
TENSOR_FMAX = fp8.E4M3_MAX * E2M1_MAX  # 2688


def e2m1_decode(code: np.ndarray) -> np.ndarray:
    """uint8 codes 0..15 -> float64 values from the bit fields."""
    c = np.asarray(code).astype(np.int64)
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 1).astype(np.float64)
    normal = (1.0 + m / 2.0) * np.exp2((e - 1).astype(np.float64))
    sub = m * 0.5
    return sign * np.where(e == 0, sub, normal)


def e2m1_encode(y: np.ndarray) -> np.ndarray:
    """float32 values -> uint8 E2M1 codes (round to nearest even, saturating to +-6).

    The magnitude is scaled into its binade and the mantissa rounded with
    ``np.rint`` (halves to even); a carry out of the mantissa moves to the next
    binade, and a carry out of the top binade (or a magnitude above 6)
    saturates.
    """
    y = np.asarray(y, np.float32).astype(np.float64)
    sign = np.where(np.signbit(y), 0x8, 0).astype(np.int64)
    a = np.abs(y)
    # binade index E: 0 for a < 1 (step 0.5), else floor(log2 a) + 1 (step 2^(E-2))
    E = np.zeros(a.shape, np.int64)
    E = np.where(a >= 1.0, 1, E)
    E = np.where(a >= 2.0, 2, E)
    E = np.where(a >= 4.0, 3, E)
    step = np.where(E == 0, 0.5, np.exp2((E - 2).astype(np.float64)))
    base = np.where(E == 0, 0.0, np.exp2((E - 1).astype(np.float64)))
    with np.errstate(invalid="ignore"):                 # non-finite quotients (S_b = 0) are replaced by the caller
        m = np.rint((a - base) / step).astype(np.int64)  # 0, 1 or 2 (2 = carry)
    code = np.where(E == 0, m, (E << 1) + m)             # a carry (m = 2) moves to the next binade: (E + 1) << 1
    code = np.where((code > 7) | (a > E2M1_MAX), 7, code)
    return (code | sign).astype(np.uint8)


def tensor_scale(x16: np.ndarray) -> np.float32:
    """``fl32(amax / 2688)`` over the whole fp16 tensor; 1 for an all-zero tensor."""
    amax = np.float32(np.max(np.abs(x16)))
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / np.float32(TENSOR_FMAX))


def quantize(x16: np.ndarray, s_t) -> tuple[np.ndarray, np.ndarray]:
    """fp16 ``[..., D]`` (blocks along the last axis) with tensor scale ``s_t`` ->
    (codes uint8 ``[..., D]`` in 0..15, block-scale bytes uint8 ``[..., D/16]``)."""
    *lead, d = x16.shape
    assert d % BLOCK == 0
    x = x16.astype(np.float32).reshape(*lead, d // BLOCK, BLOCK)
    s_t = np.float32(s_t)
    amax_b = np.max(np.abs(x), axis=-1)                                   # exact
    with np.errstate(divide="ignore", invalid="ignore"):
        sb = fp8.e4m3_encode(np.float32(amax_b / np.float32(E2M1_MAX)) / s_t)
    S_b = fp8.e4m3_decode(sb).astype(np.float32)                          # exact in fp32
    denom = (S_b * s_t).astype(np.float32)                                # fl32(S_b * s_t)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x / denom[..., None]).astype(np.float32)
    codes = e2m1_encode(q)
    codes = np.where((S_b == 0)[..., None], np.uint8(0), codes).astype(np.uint8)
    return codes.reshape(*lead, d), sb


def dequantize(codes: np.ndarray, sb: np.ndarray, s_t) -> np.ndarray:
    """``e2m1(code) * S_b * s_t`` in float64, shape of ``codes``."""
    *lead, d = codes.shape
    v = e2m1_decode(codes).reshape(*lead, d // BLOCK, BLOCK)
    S = fp8.e4m3_decode(sb).astype(np.float64)[..., None]
    return (v * S * float(np.float32(s_t))).reshape(*lead, d)
