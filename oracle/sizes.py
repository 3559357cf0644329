"""KV-cache byte accounting — oracle.

Sources:
* "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), section 1:
  KV bytes = 2 (K and V) x L x H x D x S x B x bytes per element.
* "大模型量化从0到1（十三）：KV Cache 量化" (CSDN), section 4 (the same formula with
  the KV head count, its S = 1 per-token form, the dtype table), section 5.4
  (MHA / GQA / MQA), section 10.3 (average bits with a residual window) and
  section 10.4 (scale / zero-point overhead).
* "KV Cache 量化是什么" (aigcbaba), section 3: elements per token and the FP16
  bytes per token.
"""
from __future__ import annotations

from fractions import Fraction

GROUP = 32


def kv_cache_bytes(layers: int, batch: int, seq: int, kv_heads: int, head_dim: int, bytes_per_elem) -> Fraction:
    """``2 * L * B * S * H_kv * D * b`` (b may be fractional, e.g. 1/2 for INT4)."""
    return 2 * layers * batch * seq * kv_heads * head_dim * Fraction(bytes_per_elem)


def kv_elements_per_token(layers: int, kv_heads: int, head_dim: int) -> int:
    return 2 * layers * kv_heads * head_dim


def average_bits(quantized_tokens: int, bits: int, residual_tokens: int, residual_bits: int = 16) -> Fraction:
    """Average bits per element when the newest tokens stay in high precision."""
    total = quantized_tokens + residual_tokens
    return Fraction(quantized_tokens * bits + residual_tokens * residual_bits, total)


def metadata_overhead(group_elems: int, bits: int, scale_bytes: int, zero_bytes: int) -> Fraction:
    """Metadata bytes over code bytes for one quantization group."""
    return Fraction(scale_bytes + zero_bytes) / Fraction(group_elems * bits, 8)


# ---- this library's KIVI layout (one layer) ----

def kivi_group_bytes(head_dim: int, k_bits: int, v_bits: int) -> dict:
    """Bytes of each record of one (batch, kv head, 32-token group)."""
    return {
        "k_codes": GROUP * head_dim * k_bits // 8,
        "k_meta": head_dim * 4,          # fp16 scale + fp16 zero per channel
        "v_codes": GROUP * head_dim * v_bits // 8,
        "v_meta": GROUP * 4,             # fp16 scale + fp16 zero per token
    }


def kivi_bytes_per_grouped_token(head_dim: int, k_bits: int, v_bits: int) -> Fraction:
    """Bytes read per grouped token and kv head (codes plus metadata)."""
    return Fraction(sum(kivi_group_bytes(head_dim, k_bits, v_bits).values()), GROUP)


def kivi_buffer_bytes(batch, kv_heads, head_dim, k_bits, v_bits, residual, max_tokens) -> dict:
    """Sizes of the six caller-owned buffers of a cache that holds ``max_tokens``."""
    res_cap = residual if residual > 0 else GROUP
    groups = -(-max_tokens // GROUP)
    per = kivi_group_bytes(head_dim, k_bits, v_bits)
    bh = batch * kv_heads
    out = {name: bh * groups * n for name, n in per.items()}
    out["k_res"] = bh * res_cap * head_dim * 2
    out["v_res"] = bh * res_cap * head_dim * 2
    return out


def decode_bytes_kivi(batch, kv_heads, q_heads, head_dim, k_bits, v_bits, n_grouped, n_resid) -> int:
    """Algorithmic bytes one decode-attention call must move.

    Every grouped token's codes and metadata, every residual token's fp16 K and
    V, the fp16 query and the fp16 output.
    """
    per_tok = kivi_bytes_per_grouped_token(head_dim, k_bits, v_bits)
    bh = batch * kv_heads
    grouped = per_tok * n_grouped * bh
    resid = n_resid * head_dim * 2 * 2 * bh
    qo = 2 * batch * q_heads * head_dim * 2
    return int(grouped + resid + qo)


def decode_bytes_fp8(batch, kv_heads, q_heads, head_dim, seq_len, blocks_per_seq) -> int:
    """Algorithmic bytes of one FP8 paged decode call: K and V bytes, the block table, q and out."""
    kv = 2 * batch * kv_heads * seq_len * head_dim
    table = batch * blocks_per_seq * 4
    qo = 2 * batch * q_heads * head_dim * 2
    return kv + table + qo
