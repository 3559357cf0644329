"""KIVI asymmetric group quantization and its streaming cache — oracle.

Source: "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), sections
3.1-3.4: keys are quantized per channel and values per token, in groups of 32
tokens, 2 or 4 bits, with the newest R = 128 tokens kept in fp16; when the
residual window holds R tokens it is quantized as a whole into the grouped
region and emptied. The affine form (scale, zero point, dequantize
``x_hat = (q - z) * s``) is the one of "大模型量化从0到1（十三）：KV Cache 量化"
(CSDN), section 10; KIVI's zero point is the group minimum, so
``x_hat = code * s + min``.

Arithmetic of one group x_0..x_{n-1} (fp16 values, b bits), exactly as stated
for the method (IEEE fp32, round-to-nearest-even, no fused operations):

1. ``mn = min x``, ``mx = max x`` (exact); a zero minimum is stored as +0.
2. ``s32 = fl32(fl32(mx - mn) / (2^b - 1))``; the stored scale is
   ``s16 = fp16(s32)`` and the stored zero point is ``z16 = mn`` (exact).
3. ``code_i = clamp(rint(fl32(fl32(x_i - z16) / s16)), 0, 2^b - 1)``, with rint
   rounding half to even; when ``s16 == 0`` every code is 0.
4. Dequantize: ``x_hat_i = code_i * s16 + z16`` (exact in float64).

Readings where the pages are silent: the codes are formed with the stored fp16
scale (so that the stored pair reproduces the group min and max), the value
group spans the whole head dimension of one token, and the prefill leaves
between R - G + 1 and R tokens in the residual window (R > 0) so that every
group covers tokens [32 g, 32 g + 32).
"""
from __future__ import annotations

import numpy as np

GROUP = 32


def quantize_groups(x16: np.ndarray, bits: int):
    """Quantize each group along the last axis.

    x16: fp16 array ``[..., n]``. Returns ``codes`` uint8 ``[..., n]``,
    ``scale`` fp16 ``[...]`` and ``zero`` fp16 ``[...]``.
    """
    assert x16.dtype == np.float16 and bits in (2, 4)
    x = x16.astype(np.float32)
    levels = np.float32(2 ** bits - 1)
    mn = x.min(axis=-1) + np.float32(0.0)          # -0 -> +0
    mx = x.max(axis=-1)
    s32 = (mx - mn) / levels                       # fp32 sub, fp32 div
    s16 = s32.astype(np.float16)                   # round to nearest even
    z16 = mn.astype(np.float16)                    # exact: mn is an fp16 value
    sf = s16.astype(np.float32)[..., None]
    diff = x - z16.astype(np.float32)[..., None]   # fp32 sub
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = diff / sf                          # fp32 div
    codes = np.clip(np.rint(ratio), 0, levels)
    codes = np.where(sf == 0, 0, codes).astype(np.uint8)
    return codes, s16, z16


def dequantize(codes: np.ndarray, scale16: np.ndarray, zero16: np.ndarray, axis_len_last: bool = True):
    """``x_hat = code * s + z`` in float64; scale/zero broadcast over the last axis."""
    return codes.astype(np.float64) * scale16.astype(np.float64)[..., None] + zero16.astype(np.float64)[..., None]


def quantize_key_groups(k16: np.ndarray, bits: int):
    """Keys ``[..., ng*32, D]`` -> per-channel groups of 32 tokens.

    Returns codes uint8 ``[..., ng, 32, D]`` and scale/zero fp16 ``[..., ng, D]``.
    """
    *lead, t, d = k16.shape
    assert t % GROUP == 0
    ng = t // GROUP
    grouped = k16.reshape(*lead, ng, GROUP, d)
    per_channel = np.swapaxes(grouped, -1, -2)          # [..., ng, D, 32]
    codes, s, z = quantize_groups(per_channel, bits)
    return np.swapaxes(codes, -1, -2), s, z


def quantize_value_tokens(v16: np.ndarray, bits: int):
    """Values ``[..., ng*32, D]`` -> one group per token over its D channels.

    Returns codes uint8 ``[..., ng, 32, D]`` and scale/zero fp16 ``[..., ng, 32]``.
    """
    *lead, t, d = v16.shape
    assert t % GROUP == 0
    ng = t // GROUP
    codes, s, z = quantize_groups(v16, bits)
    return (codes.reshape(*lead, ng, GROUP, d), s.reshape(*lead, ng, GROUP), z.reshape(*lead, ng, GROUP))


def prefill_split(seq_len: int, residual: int) -> tuple[int, int]:
    """(tokens in the grouped region, tokens in the fp16 window) after a prefill."""
    if residual > 0:
        grouped = GROUP * (-(-max(seq_len - residual, 0) // GROUP))
    else:
        grouped = GROUP * (seq_len // GROUP)
    return grouped, seq_len - grouped


class KiviCache:
    """The streaming KIVI cache of one layer, held as logical (unpacked) arrays.

    Grouped region: ``k_codes/v_codes`` uint8 ``[B, H, ng, 32, D]``,
    ``k_scale/k_zero`` fp16 ``[B, H, ng, D]``, ``v_scale/v_zero`` fp16
    ``[B, H, ng, 32]``. Residual window: fp16 ``[B, H, n_resid, D]``, oldest first.
    """

    def __init__(self, batch, kv_heads, head_dim, k_bits=2, v_bits=2, residual=128, max_tokens=None):
        assert residual % GROUP == 0
        self.B, self.H, self.D = batch, kv_heads, head_dim
        self.k_bits, self.v_bits, self.R = k_bits, v_bits, residual
        self.res_cap = residual if residual > 0 else GROUP
        self.max_tokens = max_tokens
        z8 = np.zeros((batch, kv_heads, 0, GROUP, head_dim), np.uint8)
        self.k_codes, self.v_codes = z8, z8.copy()
        self.k_scale = np.zeros((batch, kv_heads, 0, head_dim), np.float16)
        self.k_zero = self.k_scale.copy()
        self.v_scale = np.zeros((batch, kv_heads, 0, GROUP), np.float16)
        self.v_zero = self.v_scale.copy()
        self.k_res = np.zeros((batch, kv_heads, 0, head_dim), np.float16)
        self.v_res = self.k_res.copy()

    @property
    def n_grouped(self) -> int:
        return self.k_codes.shape[2] * GROUP

    @property
    def n_resid(self) -> int:
        return self.k_res.shape[2]

    def _add_groups(self, k16, v16):
        kc, ks, kz = quantize_key_groups(k16, self.k_bits)
        vc, vs, vz = quantize_value_tokens(v16, self.v_bits)
        self.k_codes = np.concatenate([self.k_codes, kc], axis=2)
        self.k_scale = np.concatenate([self.k_scale, ks], axis=2)
        self.k_zero = np.concatenate([self.k_zero, kz], axis=2)
        self.v_codes = np.concatenate([self.v_codes, vc], axis=2)
        self.v_scale = np.concatenate([self.v_scale, vs], axis=2)
        self.v_zero = np.concatenate([self.v_zero, vz], axis=2)

    def prefill(self, k16, v16):
        """Start the cache from ``S`` tokens: fp16 ``[B, H, S, D]`` each."""
        s = k16.shape[2]
        if self.max_tokens is not None and s > self.max_tokens:
            raise ValueError("capacity")
        self.__init__(self.B, self.H, self.D, self.k_bits, self.v_bits, self.R, self.max_tokens)
        ng_tok, _ = prefill_split(s, self.R)
        self._add_groups(k16[:, :, :ng_tok], v16[:, :, :ng_tok])
        self.k_res = k16[:, :, ng_tok:].copy()
        self.v_res = v16[:, :, ng_tok:].copy()

    def flush(self):
        """Quantize the oldest whole groups of the window and keep the rest."""
        n = GROUP * (self.n_resid // GROUP)
        if n == 0:
            return
        self._add_groups(self.k_res[:, :, :n], self.v_res[:, :, :n])
        self.k_res = self.k_res[:, :, n:].copy()
        self.v_res = self.v_res[:, :, n:].copy()

    def append(self, k_new16, v_new16):
        """One decode step's token, fp16 ``[B, H, D]`` each (section 3.2's order)."""
        if self.max_tokens is not None and self.n_grouped + self.n_resid + 1 > self.max_tokens:
            raise ValueError("capacity")
        if self.n_resid == self.res_cap:
            self.flush()
        self.k_res = np.concatenate([self.k_res, k_new16[:, :, None]], axis=2)
        self.v_res = np.concatenate([self.v_res, v_new16[:, :, None]], axis=2)
        if self.R == 0 and self.n_resid == GROUP:
            self.flush()

    # ---- dequantized views (float64) ----
    def keys_hat(self, b, h):
        """All tokens of (b, h): grouped region then residual, float64 ``[T, D]``."""
        kc = self.k_codes[b, h].astype(np.float64)                  # [ng, 32, D]
        kh = kc * self.k_scale[b, h].astype(np.float64)[:, None, :] + self.k_zero[b, h].astype(np.float64)[:, None, :]
        return np.concatenate([kh.reshape(-1, self.D), self.k_res[b, h].astype(np.float64)], axis=0)

    def values_hat(self, b, h):
        vc = self.v_codes[b, h].astype(np.float64)                  # [ng, 32, D]
        vh = vc * self.v_scale[b, h].astype(np.float64)[:, :, None] + self.v_zero[b, h].astype(np.float64)[:, :, None]
        return np.concatenate([vh.reshape(-1, self.D), self.v_res[b, h].astype(np.float64)], axis=0)
