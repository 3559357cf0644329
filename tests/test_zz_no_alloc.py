"""kv_decode_attention_noalloc: decode attention for callers that cannot allocate
device memory (for example a serving engine whose device memory is all handed
to a fixed KV-block pool, or a plugin whose host framework forbids cudaMalloc
while a step runs). It must give what kv_decode_attention gives, and stay
within the attention bars of the float64 oracle, on consecutive calls that
share the library's fixed scratch array, for both decode kernels (query heads
per kv head above 4, and at most 4) and for the stream-K cut that covers more
(batch row, kv head) pairs than the GPU keeps resident; it must refuse shapes
whose scratch would not fit.

This file is collected last on purpose; it works alone in a fresh process and
after the other tests.
"""
import numpy as np
import pytest

from oracle.attention import default_scale
from quantized_kv_cache_quant_gb300 import workloads

from kvq_helpers import assert_attention_close, dev, host, oracle_attention, oracle_cache

pytestmark = pytest.mark.gpu


def _sample_heads(b, hq, n, seed):
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (b - 1, hq - 1)}
    while len(picks) < min(n, b * hq):
        picks.add((int(rng.integers(b)), int(rng.integers(hq))))
    return sorted(picks)


@pytest.mark.parametrize("b,hkv,hq,d,s,kb,vb,seed", [
    (4, 4, 32, 128, 32 * 50 + 77, 2, 2, 123),      # 8 query heads per kv head
    (3, 8, 8, 128, 32 * 21 + 128, 2, 2, 5),        # one query head per kv head (swapped-operand kernel)
    (2, 4, 16, 64, 32 * 33 + 45, 4, 2, 6),         # 4 query heads per kv head (swapped-operand kernel)
    (64, 16, 32, 64, 32 * 37 + 119, 2, 2, 21),     # 1024 pairs: the stream-K cut, more pairs than resident blocks
])
def test_noalloc_matches_workspace_call_and_oracle(b, hkv, hq, d, s, kb, vb, seed):
    import torch
    from quantized_kv_cache_quant_gb300 import kvq

    x = workloads.make_inputs(b, hkv, hq, d, s, 2, seed)
    cache = kvq.KiviCache(b, hkv, hq, d, kb, vb, 128, s + 2)
    cache.prefill(dev(x.k), dev(x.v))
    oc = oracle_cache(dict(k_bits=kb, v_bits=vb, residual=128, max_tokens=s + 2), x.k, x.v)
    heads = None if b * hq <= 256 else _sample_heads(b, hq, 64, seed)
    kvq.kv_decode_noalloc_status(clear=True)
    for step in range(2):                        # two calls in a row on the shared scratch array
        if step:
            cache.append(dev(x.k_new[step]), dev(x.v_new[step]))
            oc.append(x.k_new[step], x.v_new[step])
        q = dev(x.q[step])
        same = host(cache.decode(q)).astype(np.float64)
        out = torch.full((b, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        kvq.kv_decode_attention_noalloc(cache.desc, q, out, True, 0.0)
        got = host(out)
        assert_attention_close(got, same)
        ref = oracle_attention(oc, x.q[step], default_scale(d), heads)
        assert_attention_close(got, ref, heads)
    # fp16 output through the same call
    out16 = torch.empty((b, hq, d), dtype=torch.float16, device="cuda")
    kvq.kv_decode_attention_noalloc(cache.desc, q, out16, False, 0.0)
    assert_attention_close(host(out16).astype(np.float64), ref, heads, fp16_out=True)
    assert kvq.kv_decode_noalloc_status() == 0


def test_noalloc_status_word_is_read_and_cleared():
    from quantized_kv_cache_quant_gb300 import kvq

    assert kvq.kv_decode_noalloc_status(clear=True) == 0
    assert kvq.kv_decode_noalloc_status() == 0


def test_noalloc_rejects_oversized_scratch():
    from quantized_kv_cache_quant_gb300 import kvq

    # 1024 x 64 query heads x (D + 2) floats already exceed 16 MiB for one split
    cfg = kvq.make_config(1024, 8, 64, 128, 2, 2, 128, 4096)
    fake = 1 << 20                               # validation fails before any device access
    cache = kvq.kivi_cache_init(cfg, [fake * (i + 1) for i in range(6)])
    cache.n_grouped, cache.n_resid = 1024, 64
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_decode_attention_noalloc(cache, fake, fake, True, 0.0)
    assert e.value.name == "KVQ_ERR_CAPACITY"
