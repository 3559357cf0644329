"""Byte layout of the packed KIVI cache — oracle side.

Written from the format specification in ``include/kvq.h`` (section "Grouped
region layout"); it shares no code with the CUDA library. The layout is this
library's own choice (the pages fix the codes and their meaning, not their
placement in memory).

Per (batch, kv head, group of 32 tokens) there are four records:

* key codes   : 32 lanes x W words (W = D/16 at 2 bits, D/8 at 4 bits), u32
* key meta    : (D/16) x 4 records of 16 bytes:
                {s[d0], s[d0+1], s[d0+8], s[d0+9], z[d0], z[d0+1], z[d0+8], z[d0+9]}
                (fp16) with d0 = 16*ks + 2*tig, record index ks*4 + tig
* value codes : 32 lanes x W words, u32
* value meta  : 4 x 16 bytes of scales then 4 x 16 bytes of zeros; record tig
                holds tokens {2tig, 2tig+1, 8+2tig, 9+2tig, 16+2tig, 17+2tig,
                24+2tig, 25+2tig}

Code words. A lane is ``lane = 4*g + tig`` (g in 0..7, tig in 0..3). Each
32-bit word carries codes for one pair of elements in its two 16-bit halves
(low half: first element of the pair, high half: second element). For a
pair ``(ks, r, nt)``:

* keys   : elements are channels ``d0 = 16*ks + 8*r + 2*tig`` and ``d0+1`` of
           token ``8*nt + g`` (nt in 0..3, ks in 0..D/16-1);
* values : elements are tokens ``t0 = 16*ks + 8*r + 2*tig`` and ``t0+1`` of
           channel ``8*nt + g`` (nt in 0..D/8-1, ks in 0..1).

With ``NQ`` = 1 for keys and D/32 for values:

* 2 bits: word ``u = ks*NQ + nt//4``, field ``f = (4*r + nt%4 + 1) mod 8`` at
  bits ``[2f, 2f+2)`` of each half (the order in which the unshifted word,
  its shifts by 4 either way and its per-half byte swap expose the fields);
* 4 bits: word ``u = (2*ks + r)*NQ + nt//4``, field ``f = nt%4`` at bits
  ``[4f, 4f+4)`` of each half.

Word ``u`` of lane ``lane`` is stored at u32 index ``(u//4)*128 + lane*4 + u%4``.
"""
from __future__ import annotations

import numpy as np

GROUP = 32


def code_words_per_lane(head_dim: int, bits: int) -> int:
    return head_dim // 16 if bits == 2 else head_dim // 8


def _word_address(lane: int, u: int) -> int:
    return (u // 4) * 128 + lane * 4 + (u % 4)


def _place(words, lane, u, f, bits, lo_code, hi_code):
    shift = bits * f
    words[..., _word_address(lane, u)] |= (lo_code.astype(np.uint32) << shift) | (hi_code.astype(np.uint32) << (16 + shift))


def pack_key_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes uint8 ``[..., 32, D]`` (token, channel) -> uint8 ``[..., 32*W*4]``."""
    *lead, t, d = codes.shape
    assert t == GROUP
    w = code_words_per_lane(d, bits)
    words = np.zeros((*lead, 32 * w), np.uint32)
    for lane in range(32):
        g, tig = lane // 4, lane % 4
        for ks in range(d // 16):
            for r in range(2):
                d0 = 16 * ks + 8 * r + 2 * tig
                for nt in range(4):
                    tok = 8 * nt + g
                    if bits == 2:
                        u, f = ks, (4 * r + nt % 4 + 1) % 8
                    else:
                        u, f = 2 * ks + r, nt % 4
                    _place(words, lane, u, f, bits, codes[..., tok, d0], codes[..., tok, d0 + 1])
    return words.view(np.uint8).reshape(*lead, -1)


def pack_value_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes uint8 ``[..., 32, D]`` (token, channel) -> uint8 ``[..., 32*W*4]``."""
    *lead, t, d = codes.shape
    assert t == GROUP
    w = code_words_per_lane(d, bits)
    nq = d // 32
    words = np.zeros((*lead, 32 * w), np.uint32)
    for lane in range(32):
        g, tig = lane // 4, lane % 4
        for ks in range(2):
            for r in range(2):
                t0 = 16 * ks + 8 * r + 2 * tig
                for nt in range(d // 8):
                    ch = 8 * nt + g
                    if bits == 2:
                        u, f = ks * nq + nt // 4, (4 * r + nt % 4 + 1) % 8
                    else:
                        u, f = (2 * ks + r) * nq + nt // 4, nt % 4
                    _place(words, lane, u, f, bits, codes[..., t0, ch], codes[..., t0 + 1, ch])
    return words.view(np.uint8).reshape(*lead, -1)


def pack_key_meta(scale16: np.ndarray, zero16: np.ndarray) -> np.ndarray:
    """scale/zero fp16 ``[..., D]`` -> uint8 ``[..., 4*D]``."""
    *lead, d = scale16.shape
    out = np.zeros((*lead, d // 16, 4, 8), np.uint16)
    s, z = scale16.view(np.uint16), zero16.view(np.uint16)
    for ks in range(d // 16):
        for tig in range(4):
            d0 = 16 * ks + 2 * tig
            chans = [d0, d0 + 1, d0 + 8, d0 + 9]
            for j, c in enumerate(chans):
                out[..., ks, tig, j] = s[..., c]
                out[..., ks, tig, 4 + j] = z[..., c]
    return out.view(np.uint8).reshape(*lead, -1)


def pack_value_meta(scale16: np.ndarray, zero16: np.ndarray) -> np.ndarray:
    """scale/zero fp16 ``[..., 32]`` (per token) -> uint8 ``[..., 128]``."""
    *lead, t = scale16.shape
    assert t == GROUP
    out = np.zeros((*lead, 2, 4, 8), np.uint16)
    s, z = scale16.view(np.uint16), zero16.view(np.uint16)
    for tig in range(4):
        toks = [2 * tig, 2 * tig + 1, 8 + 2 * tig, 9 + 2 * tig, 16 + 2 * tig, 17 + 2 * tig, 24 + 2 * tig, 25 + 2 * tig]
        for j, tk in enumerate(toks):
            out[..., 0, tig, j] = s[..., tk]
            out[..., 1, tig, j] = z[..., tk]
    return out.view(np.uint8).reshape(*lead, -1)


def pack_cache(cache) -> dict:
    """All four grouped records of an ``oracle.kivi.KiviCache``: uint8 ``[B, H, ng, bytes]``."""
    return {
        "k_codes": pack_key_codes(cache.k_codes, cache.k_bits),
        "k_meta": pack_key_meta(cache.k_scale, cache.k_zero),
        "v_codes": pack_value_codes(cache.v_codes, cache.v_bits),
        "v_meta": pack_value_meta(cache.v_scale, cache.v_zero),
    }


# ---------------------------------------------------------------------------
# FP8 paged blocks: byte order inside one (block, kv head) of 16 tokens x D
# ---------------------------------------------------------------------------
# From the pool specification in ``include/kvq.h``: each lane = 4*g + tig owns
# D/2 bytes (D/4 byte pairs); byte p of lane l's stream is stored at byte
# ((p//16)*32 + l)*16 + p%16 of the block.
#   keys   : pair i = (nt*(D//16) + ks)*2 + r holds channels d0 = 16ks + 8r + 2tig
#            and d0+1 of token 8nt + g (nt < 2);
#   values : pair i = nt*2 + r holds tokens t0 = 8r + 2tig and t0+1 of channel
#            8nt + g (nt < D/8).

def fp8_block_order(head_dim: int, value_layout: int) -> np.ndarray:
    """perm[storage_byte] = index into the natural row-major [16, D] block.

    value_layout 0 (keys) and 1 (values) hold byte pairs (m16n8k16 fragments
    after an exact fp8 -> fp16 conversion); value_layout 2 (keys read by FP8
    tensor cores) holds 4-byte words: word w = (nt * (D/32) + kk) * 2 + r of
    lane (g, tig) is channels 32*kk + 16*r + 4*tig .. +3 of token 8*nt + g.
    """
    d = head_dim
    perm = np.full(16 * d, -1, np.int64)
    for lane in range(32):
        g, tig = lane // 4, lane % 4
        elems = []                                   # (token, channel) of stream bytes 0, 1, 2, ...
        if value_layout == 2:
            for w in range(d // 8):
                nt, rem = w // (d // 16), w % (d // 16)
                kk, r = rem // 2, rem % 2
                c0 = 32 * kk + 16 * r + 4 * tig
                elems += [(8 * nt + g, c0 + e) for e in range(4)]
        else:
            for i in range(d // 4):
                if value_layout == 1:
                    nt, r = i // 2, i % 2
                    t0 = 8 * r + 2 * tig
                    elems += [(t0, 8 * nt + g), (t0 + 1, 8 * nt + g)]
                else:
                    nt, rem = i // (d // 8), i % (d // 8)
                    ks, r = rem // 2, rem % 2
                    d0 = 16 * ks + 8 * r + 2 * tig
                    elems += [(8 * nt + g, d0), (8 * nt + g, d0 + 1)]
        for p, (tok, ch) in enumerate(elems):
            perm[((p // 16) * 32 + lane) * 16 + p % 16] = tok * d + ch
    assert np.all(perm >= 0)
    return perm


def fp8_pack_pool(natural_pool: np.ndarray, value_layout: int) -> np.ndarray:
    """[nb, H, 16, D] natural blocks -> [nb, H, 16*D] in fragment byte order."""
    nb, h, bs, d = natural_pool.shape
    assert bs == 16
    perm = fp8_block_order(d, value_layout)
    return natural_pool.reshape(nb, h, bs * d)[:, :, perm]


def fp8_unpack_pool(packed_pool: np.ndarray, head_dim: int, value_layout: int) -> np.ndarray:
    """Inverse of ``fp8_pack_pool``."""
    nb, h, n = packed_pool.shape
    perm = fp8_block_order(head_dim, value_layout)
    out = np.empty_like(packed_pool)
    out[:, :, perm] = packed_pool
    return out.reshape(nb, h, 16, head_dim)


# ---------------------------------------------------------------------------
# NVFP4 paged blocks: one (block, kv head) record of 16 tokens x D holds
# 8*D bytes of 4-bit codes, then D bytes of E4M3 block scales
# (specification in ``include/kvq.h``, section "NVFP4 paged cache").
#   keys   : lane = 4g + tig owns 4*KS code bytes (KS = D/16); its byte
#            i = (nt*KS + ks)*2 + r holds channels c0 = 16ks + 8r + 2tig (low
#            nibble) and c0 + 1 (high nibble) of token 8nt + g (nt < 2);
#            scale byte g*2*KS + nt*KS + ks is the scale of token 8nt + g,
#            channels 16ks .. 16ks + 15.
#   values : lane owns D/4 code bytes; its byte i = nt*2 + r holds tokens
#            t0 = 8r + 2tig (low nibble) and t0 + 1 (high nibble) of channel
#            8nt + g (nt < D/8); scale byte ((tig*2 + r)*(D/16) + j)*2 + e is
#            the scale of token 8r + 2tig + e, channels 16j .. 16j + 15.
# Byte p of a lane's code stream is stored at ((p//16)*32 + lane)*16 + p%16.
# ---------------------------------------------------------------------------

def nvfp4_pack_record(codes: np.ndarray, scales: np.ndarray, role: int) -> np.ndarray:
    """One block: codes uint8 ``[16, D]`` (0..15), scales uint8 ``[16, D/16]`` -> uint8 ``[9*D]``."""
    t, d = codes.shape
    assert t == 16
    ks_n = d // 16
    out = np.zeros(9 * d, np.uint8)
    for lane in range(32):
        g, tig = lane // 4, lane % 4
        stream = []
        if role == 0:
            for nt in range(2):
                for ks in range(ks_n):
                    for r in range(2):
                        c0 = 16 * ks + 8 * r + 2 * tig
                        tok = 8 * nt + g
                        stream.append(int(codes[tok, c0]) | (int(codes[tok, c0 + 1]) << 4))
        else:
            for nt in range(d // 8):
                for r in range(2):
                    t0 = 8 * r + 2 * tig
                    ch = 8 * nt + g
                    stream.append(int(codes[t0, ch]) | (int(codes[t0 + 1, ch]) << 4))
        for p, byte in enumerate(stream):
            out[((p // 16) * 32 + lane) * 16 + p % 16] = byte
    sc = out[8 * d:]
    if role == 0:
        for g in range(8):
            for nt in range(2):
                for ks in range(ks_n):
                    sc[g * 2 * ks_n + nt * ks_n + ks] = scales[8 * nt + g, ks]
    else:
        for tig in range(4):
            for r in range(2):
                for j in range(ks_n):
                    for e in range(2):
                        sc[((tig * 2 + r) * ks_n + j) * 2 + e] = scales[8 * r + 2 * tig + e, j]
    return out


def nvfp4_pack_pool(codes_pool: np.ndarray, scales_pool: np.ndarray, role: int) -> np.ndarray:
    """Natural blocks codes ``[nb, H, 16, D]``, scales ``[nb, H, 16, D/16]`` -> ``[nb, H, 9*D]``."""
    nb, h, _, d = codes_pool.shape
    out = np.zeros((nb, h, 9 * d), np.uint8)
    for b in range(nb):
        for hh in range(h):
            if codes_pool[b, hh].any() or scales_pool[b, hh].any():
                out[b, hh] = nvfp4_pack_record(codes_pool[b, hh], scales_pool[b, hh], role)
    return out
