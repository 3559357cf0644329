"""Paged, variable-length KIVI cache — oracle (test infrastructure only).

A serving cache holds sequences of different lengths. Each sequence is a KIVI
cache of its own (keys per channel, values per token, groups of 32 tokens, an
fp16 residual window flushed when full: "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV
Cache" (aiinfraguide), section 3) whose groups are stored as blocks of a shared
pool and reached through a block table, as paged caches reach their blocks
("大模型量化从0到1（十三）：KV Cache 量化" (CSDN), section 13).

Reading (the pages combine the two ideas without a layout): one block holds one
32-token group of one sequence for every kv head; for each kv head the four
records of the contiguous cache (key codes, key meta, value codes, value meta)
sit back to back, so one group of one head is one contiguous run of bytes;
``block_table[b, g]`` is the pool block of logical group g of sequence b; each
sequence keeps its own fp16 window; every sequence follows the contiguous
cache's rules (prefill split, flush timing) on its own length. Decode attention
of sequence b runs over its grouped tokens, then its window tokens.
"""
from __future__ import annotations

import numpy as np

from . import kivi, layout


class PagedKiviCache:
    """``B`` per-sequence KIVI caches placed in pools through ``block_table [B, max_groups]``."""

    def __init__(self, batch, kv_heads, head_dim, k_bits, v_bits, residual, num_blocks, block_table):
        self.B, self.H, self.D = batch, kv_heads, head_dim
        self.k_bits, self.v_bits, self.R = k_bits, v_bits, residual
        self.num_blocks = num_blocks
        self.table = np.asarray(block_table, np.int32)
        self.seqs = [kivi.KiviCache(1, kv_heads, head_dim, k_bits, v_bits, residual) for _ in range(batch)]

    def prefill(self, k16, v16, seq_lens):
        """k16, v16: fp16 ``[B, H, S_max, D]``; sequence b uses its first seq_lens[b] tokens."""
        for b, c in enumerate(self.seqs):
            n = int(seq_lens[b])
            c.prefill(k16[b:b + 1, :, :n], v16[b:b + 1, :, :n])

    def append(self, k_new16, v_new16):
        """One token for every sequence: fp16 ``[B, H, D]``."""
        for b, c in enumerate(self.seqs):
            c.append(k_new16[b:b + 1], v_new16[b:b + 1])

    def n_grouped(self, b):
        return self.seqs[b].n_grouped

    def n_resid(self, b):
        return self.seqs[b].n_resid

    def pools(self) -> dict:
        """The four record pools, uint8 ``[num_blocks, H, bytes]``; blocks no group uses stay 0."""
        out = {name: np.zeros((self.num_blocks, self.H, nbytes), np.uint8)
               for name, nbytes in self.record_bytes().items()}
        for b, c in enumerate(self.seqs):
            if c.n_grouped == 0:
                continue
            packed = layout.pack_cache(c)                  # name -> [1, H, ng, bytes]
            for name, rec in packed.items():
                for g in range(rec.shape[2]):
                    out[name][self.table[b, g]] = rec[0, :, g]
        return out

    ORDER = ("k_codes", "k_meta", "v_codes", "v_meta")

    def pool(self) -> np.ndarray:
        """The block pool, uint8 ``[num_blocks, H, sum of record bytes]``: per
        (block, kv head) the four records in ORDER, back to back."""
        p = self.pools()
        return np.concatenate([p[name] for name in self.ORDER], axis=2)

    def record_offsets(self) -> dict:
        """Byte offset of each record inside one (block, kv head) entry of the pool."""
        out, off = {}, 0
        for name in self.ORDER:
            out[name] = off
            off += self.record_bytes()[name]
        return out

    def record_bytes(self) -> dict:
        """Bytes of one block of each record for one kv head (as in the contiguous cache)."""
        return {"k_codes": 32 * self.D * self.k_bits // 8, "k_meta": 4 * self.D,
                "v_codes": 32 * self.D * self.v_bits // 8, "v_meta": 128}

    def window(self, b):
        """Sequence b's fp16 window: (k, v) ``[H, n_resid, D]``."""
        c = self.seqs[b]
        return c.k_res[0], c.v_res[0]

    def keys_hat(self, b, h):
        return self.seqs[b].keys_hat(0, h)

    def values_hat(self, b, h):
        return self.seqs[b].values_hat(0, h)
