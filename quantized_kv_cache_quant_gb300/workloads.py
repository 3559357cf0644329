"""Seeded synthetic workloads shaped like the pages' decode caches.

This module only draws random numbers; it holds none of the quantization or
attention arithmetic, so both the CUDA path (tests, bench) and the CPU oracle
can take their inputs from it.

Distributions (the same for every workload):

* ``c[h, d] ~ LogNormal(0, 1)`` per (kv head, channel); two channels per kv head,
  chosen by the seeded generator, are multiplied by 10 (outlier channels: the
  per-channel structure of keys described in "4.4 KV Cache 量化：KIVI 2-bit 与
  FP8 KV Cache", section 2).
* ``K[b, h, t, d] = N(0, 1) * c[h, d]``.
* ``tau[b, h, t] ~ LogNormal(0, 0.5)`` per (batch, kv head, token) and
  ``V[b, h, t, d] = N(0, 1) * tau[b, h, t]`` (per-token structure of values,
  same section).
* ``q[step, b, hq, d] ~ N(0, 1)``.
* Decode-step tokens follow the same laws: ``k_new = N(0,1) * c``,
  ``v_new = N(0,1) * tau_new`` with a fresh ``tau_new`` per (step, b, h).

Draw order is fixed: c, outlier indices, K, tau, V, q, k_new, tau_new, v_new.
Large tensors are drawn one batch row at a time (float32 normals, then the
product is rounded to fp16), which keeps host memory bounded.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GROUP = 32  # KIVI group size in tokens


@dataclasses.dataclass(frozen=True)
class KiviWorkload:
    name: str
    batch: int
    kv_heads: int
    q_heads: int
    head_dim: int
    prefill: int          # tokens quantized by the prefill call
    decode_steps: int     # decode steps after the prefill
    k_bits: int = 2
    v_bits: int = 2
    residual: int = 128
    seed: int = 0

    @property
    def max_tokens(self) -> int:
        return self.prefill + self.decode_steps


@dataclasses.dataclass(frozen=True)
class Fp8Workload:
    name: str
    batch: int
    kv_heads: int
    q_heads: int
    head_dim: int
    context: int
    block_size: int = 16
    seed: int = 3
    fmt: str = "e4m3"          # FP8 format: "e4m3" or "e5m2"
    per_head: bool = False     # one scale per kv head instead of one per tensor
    q_fp8: bool = False        # FP8-domain attention: the query quantized to E4M3 too

    @property
    def blocks_per_seq(self) -> int:
        return -(-self.context // self.block_size)


@dataclasses.dataclass(frozen=True)
class Nvfp4Workload:
    """An NVFP4 paged cache (4-bit E2M1 values, E4M3 scale per 16 channels, fp32 tensor scale)."""
    name: str
    batch: int
    kv_heads: int
    q_heads: int
    head_dim: int
    context: int
    block_size: int = 16
    seed: int = 3

    @property
    def blocks_per_seq(self) -> int:
        return -(-self.context // self.block_size)


@dataclasses.dataclass(frozen=True)
class PagedKiviWorkload:
    """A batch of sequences of different lengths in one paged KIVI cache."""
    name: str
    batch: int
    kv_heads: int
    q_heads: int
    head_dim: int
    min_len: int          # prefill lengths are drawn uniformly from [min_len, max_len]
    max_len: int
    decode_steps: int = 1
    k_bits: int = 2
    v_bits: int = 2
    residual: int = 128
    seed: int = 5

    @property
    def max_tokens(self) -> int:
        return self.max_len + self.decode_steps

    @property
    def groups_cap(self) -> int:
        return -(-self.max_tokens // GROUP)

    @property
    def num_blocks(self) -> int:
        return self.batch * self.groups_cap


# The five workloads: a tiny correctness case, a Llama-2-7B-like MHA layer at 4K,
# a Llama-2-70B-like GQA layer at 8K (2- and 4-bit), an FP8 paged cache at 32K,
# and a 128K streaming cache with 512 decode steps.
TINY = KiviWorkload("kivi2_tiny_b1_h2_d64_s256", 1, 2, 2, 64, 256, 16, seed=0)
MHA_4K = KiviWorkload("kivi2_mha_b8_h32_d128_s4096", 8, 32, 32, 128, 4096, 1, seed=1)
GQA_8K_2BIT = KiviWorkload("kivi2_gqa8_b32_h8x64_d128_s8192", 32, 8, 64, 128, 8192, 1, seed=2)
GQA_8K_4BIT = dataclasses.replace(GQA_8K_2BIT, name="kivi4_gqa8_b32_h8x64_d128_s8192", k_bits=4, v_bits=4)
FP8_32K = Fp8Workload("fp8_e4m3_paged_b64_h8x32_d128_s32768", 64, 8, 32, 128, 32768, 16, seed=3)
# the same cache in E5M2 with one scale per kv head (the FP8 variants of the pages)
FP8_32K_E5M2_PH = dataclasses.replace(FP8_32K, name="fp8_e5m2_perhead_paged_b64_h8x32_d128_s32768", fmt="e5m2",
                                      per_head=True)
# the same cache read with the query in E4M3 (FP8-domain attention on FP8 tensor cores)
FP8_32K_QFP8 = dataclasses.replace(FP8_32K, name="fp8_e4m3_qfp8_paged_b64_h8x32_d128_s32768", q_fp8=True)
# the same cache for 8 sequences: a size an ncu capture of the quantize kernels can hold
FP8_32K_B8 = Fp8Workload("fp8_e4m3_paged_b8_h8x32_d128_s32768", 8, 8, 32, 128, 32768, 16, seed=3)
# the FP8 32K cache's inputs in NVFP4 (the 4-bit floating-point KV of Blackwell-class GPUs)
NVFP4_32K = Nvfp4Workload("nvfp4_paged_b64_h8x32_d128_s32768", 64, 8, 32, 128, 32768, 16, seed=3)
NVFP4_32K_B8 = Nvfp4Workload("nvfp4_paged_b8_h8x32_d128_s32768", 8, 8, 32, 128, 32768, 16, seed=3)
STREAM_128K = KiviWorkload("kivi2_stream_b4_h8x64_d128_s131072_512steps", 4, 8, 64, 128, 131072, 512, seed=4)
# Paged caches of the GQA 8K shape: every sequence at 8192 tokens (the cost of
# the block table against the contiguous layout), and lengths spread over
# 512 .. 16384 (the balance of the split across pairs of unequal length).
PAGED_GQA_8K = PagedKiviWorkload("kivi2_paged_b32_h8x64_d128_len8192", 32, 8, 64, 128, 8192, 8192, seed=5)
PAGED_VAR_16K = PagedKiviWorkload("kivi2_paged_b32_h8x64_d128_len512-16384", 32, 8, 64, 128, 512, 16384, seed=6)
# the same lengths with four query heads per kv head (Llama-3-8B / Mistral-7B-like heads)
PAGED_GQA4_VAR_16K = PagedKiviWorkload("kivi2_paged_b32_h8x32_d128_len512-16384", 32, 8, 32, 128, 512, 16384, seed=6)

WORKLOADS = {w.name: w for w in (TINY, MHA_4K, GQA_8K_2BIT, GQA_8K_4BIT, FP8_32K, FP8_32K_E5M2_PH, FP8_32K_QFP8,
                                  FP8_32K_B8, NVFP4_32K, NVFP4_32K_B8, STREAM_128K, PAGED_GQA_8K, PAGED_VAR_16K,
                                  PAGED_GQA4_VAR_16K)}


def _channel_scales(rng: np.random.Generator, kv_heads: int, head_dim: int) -> np.ndarray:
    c = rng.lognormal(0.0, 1.0, size=(kv_heads, head_dim)).astype(np.float32)
    for h in range(kv_heads):
        idx = rng.choice(head_dim, size=2, replace=False)
        c[h, idx] *= np.float32(10.0)
    return c


def _keys(rng, c, batch, seq):
    kv_heads, d = c.shape
    out = np.empty((batch, kv_heads, seq, d), np.float16)
    for b in range(batch):
        z = rng.standard_normal((kv_heads, seq, d), dtype=np.float32)
        z *= c[:, None, :]
        out[b] = z.astype(np.float16)
    return out


def _values(rng, batch, kv_heads, seq, d):
    tau = rng.lognormal(0.0, 0.5, size=(batch, kv_heads, seq)).astype(np.float32)
    out = np.empty((batch, kv_heads, seq, d), np.float16)
    for b in range(batch):
        z = rng.standard_normal((kv_heads, seq, d), dtype=np.float32)
        z *= tau[b][:, :, None]
        out[b] = z.astype(np.float16)
    return out


@dataclasses.dataclass
class KVInputs:
    k: np.ndarray          # fp16 [B, Hkv, S, D]
    v: np.ndarray          # fp16 [B, Hkv, S, D]
    q: np.ndarray          # fp16 [steps, B, Hq, D]
    k_new: np.ndarray      # fp16 [steps, B, Hkv, D]
    v_new: np.ndarray      # fp16 [steps, B, Hkv, D]


def make_inputs(batch: int, kv_heads: int, q_heads: int, head_dim: int, seq: int,
                steps: int, seed: int) -> KVInputs:
    """Draw one cache of ``seq`` tokens plus ``steps`` decode steps (host fp16)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    c = _channel_scales(rng, kv_heads, head_dim)
    k = _keys(rng, c, batch, seq)
    v = _values(rng, batch, kv_heads, seq, head_dim)
    q = rng.standard_normal((steps, batch, q_heads, head_dim), dtype=np.float32).astype(np.float16)
    kz = rng.standard_normal((steps, batch, kv_heads, head_dim), dtype=np.float32)
    k_new = (kz * c[None, None]).astype(np.float16)
    tau = rng.lognormal(0.0, 0.5, size=(steps, batch, kv_heads)).astype(np.float32)
    vz = rng.standard_normal((steps, batch, kv_heads, head_dim), dtype=np.float32)
    v_new = (vz * tau[..., None]).astype(np.float16)
    return KVInputs(k, v, q, k_new, v_new)


def kivi_inputs(w: KiviWorkload, seq: Optional[int] = None, steps: Optional[int] = None) -> KVInputs:
    return make_inputs(w.batch, w.kv_heads, w.q_heads, w.head_dim,
                       w.prefill if seq is None else seq,
                       w.decode_steps if steps is None else steps, w.seed)


def fp8_inputs(w, context: Optional[int] = None):
    """K, V fp16 [B, Hkv, S, D], q fp16 [B, Hq, D] and a randomly permuted block table."""
    s = w.context if context is None else context
    x = make_inputs(w.batch, w.kv_heads, w.q_heads, w.head_dim, s, 1, w.seed)
    nb = -(-s // w.block_size)
    table = block_table(w.batch, nb, w.seed + 1000)
    return x.k, x.v, x.q[0], table


def block_table(batch: int, blocks_per_seq: int, seed: int) -> np.ndarray:
    """A random permutation of ``batch * blocks_per_seq`` physical blocks, int32 [B, nb]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(batch * blocks_per_seq).astype(np.int32)
    return perm.reshape(batch, blocks_per_seq)


def paged_lengths(batch: int, min_len: int, max_len: int, seed: int) -> np.ndarray:
    """Prefill lengths, int32 [B], uniform on [min_len, max_len]."""
    rng = np.random.Generator(np.random.PCG64(seed + 2000))
    return rng.integers(min_len, max_len + 1, size=batch).astype(np.int32)


def paged_inputs(w: PagedKiviWorkload, steps: Optional[int] = None):
    """(inputs [B, Hkv, max_len, D] of which sequence b uses its first lengths[b]
    tokens, the lengths, and a random permutation of every pool block as the
    block table int32 [B, groups_cap])."""
    x = make_inputs(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.max_len,
                    w.decode_steps if steps is None else steps, w.seed)
    lens = paged_lengths(w.batch, w.min_len, w.max_len, w.seed)
    return x, lens, block_table(w.batch, w.groups_cap, w.seed + 1000)
