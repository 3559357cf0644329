"""Algorithmic byte counts of the library's calls (the roofline numerators).

A call's algorithmic bytes are the bytes it must move at minimum: every byte
of the cache it reads once, its inputs and its outputs. Grouped KIVI tokens
cost their packed codes plus the fp16 scale/zero-point metadata (per kv head
and token at D = 128: 32 + 16 + 32 + 4 = 84 bytes at 2 bits, 148 at 4 bits);
window tokens cost their fp16 K and V (512 bytes at D = 128).
"""
from __future__ import annotations

GROUP = 32


def grouped_bytes_per_token(head_dim: int, k_bits: int, v_bits: int) -> float:
    per_group = GROUP * head_dim * k_bits // 8 + 4 * head_dim + GROUP * head_dim * v_bits // 8 + 4 * GROUP
    return per_group / GROUP


def kivi_decode_bytes(batch, kv_heads, q_heads, head_dim, k_bits, v_bits, n_grouped, n_resid, out_bytes=4) -> int:
    """One kv_decode_attention call: packed groups + fp16 window + q (fp16) + out."""
    bh = batch * kv_heads
    grouped = int(grouped_bytes_per_token(head_dim, k_bits, v_bits) * n_grouped) * bh
    window = n_resid * head_dim * 2 * 2 * bh
    q = batch * q_heads * head_dim * 2
    out = batch * q_heads * head_dim * out_bytes
    return grouped + window + q + out


def kivi_paged_decode_bytes(kv_heads, q_heads, head_dim, k_bits, v_bits, n_grouped, n_resid, out_bytes=4) -> int:
    """One kv_paged_decode_attention call over sequences holding n_grouped[b]
    grouped and n_resid[b] window tokens: each sequence's records and window, its
    block-table entries (int32 per group), q and out."""
    total = 0
    for ng, nr in zip(n_grouped, n_resid):
        total += kivi_decode_bytes(1, kv_heads, q_heads, head_dim, k_bits, v_bits, ng, nr, out_bytes)
        total += 4 * (ng // GROUP)
    return total


def kivi_append_bytes(batch, kv_heads, head_dim) -> int:
    """kv_append_token without a flush: read k_new, v_new; write them into the window."""
    return 2 * 2 * batch * kv_heads * head_dim * 2


def kivi_flush_bytes(batch, kv_heads, head_dim, k_bits, v_bits, n_tokens) -> int:
    """Quantizing n_tokens window tokens: read fp16 K and V, write the packed groups."""
    bh = batch * kv_heads
    read = n_tokens * head_dim * 2 * 2 * bh
    written = int(grouped_bytes_per_token(head_dim, k_bits, v_bits) * n_tokens) * bh
    return read + written


def kivi_prefill_bytes(batch, kv_heads, head_dim, k_bits, v_bits, n_grouped, n_resid) -> int:
    """kv_quant_prefill: read all fp16 K and V, write packed groups and the window copy."""
    bh = batch * kv_heads
    read = (n_grouped + n_resid) * head_dim * 2 * 2 * bh
    written = int(grouped_bytes_per_token(head_dim, k_bits, v_bits) * n_grouped) * bh + n_resid * head_dim * 4 * bh
    return read + written


def fp8_decode_bytes(batch, kv_heads, q_heads, head_dim, seq_len, blocks_per_seq, out_bytes=4) -> int:
    """One fp8_decode_attention call: K and V bytes, the block table, q and out."""
    kv = 2 * batch * kv_heads * seq_len * head_dim
    return kv + batch * blocks_per_seq * 4 + batch * q_heads * head_dim * (2 + out_bytes)


def fp8_quantize_bytes(batch, kv_heads, seq_len, head_dim, dynamic: bool) -> int:
    """One fp8_kv_quantize call: (amax pass +) cast pass over fp16 x, FP8 bytes written."""
    n = batch * kv_heads * seq_len * head_dim
    return n * 2 * (2 if dynamic else 1) + n


def nvfp4_record_bytes_per_token(head_dim) -> int:
    """NVFP4 bytes of one token of one kv head: D/2 code bytes and D/16 scale bytes."""
    return head_dim // 2 + head_dim // 16


def nvfp4_decode_bytes(batch, kv_heads, q_heads, head_dim, seq_len, blocks_per_seq, out_bytes=4) -> int:
    """One nvfp4_decode_attention call: K and V records, the block table, q and out."""
    kv = 2 * batch * kv_heads * seq_len * nvfp4_record_bytes_per_token(head_dim)
    return kv + batch * blocks_per_seq * 4 + batch * q_heads * head_dim * (2 + out_bytes)


def nvfp4_quantize_bytes(batch, kv_heads, seq_len, head_dim, dynamic: bool) -> int:
    """One nvfp4_kv_quantize call: (amax pass +) cast pass over fp16 x, records written."""
    n = batch * kv_heads * seq_len
    return n * head_dim * 2 * (2 if dynamic else 1) + n * nvfp4_record_bytes_per_token(head_dim)
