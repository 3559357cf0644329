"""kv_decode_attention_noalloc: decode attention for callers that cannot allocate
device memory (for example a serving engine whose device memory is all handed
to a fixed KV-block pool, or a plugin whose host framework forbids cudaMalloc
while a step runs). It must give what kv_decode_attention gives, within the
attention tolerance of the parity tests, on consecutive calls that share the
library's fixed scratch array, and refuse shapes whose scratch would not fit.

This file is collected last on purpose; it works alone in a fresh process and
after the other tests.
"""
import numpy as np
import pytest

from quantized_kv_cache_quant_gb300 import workloads

from kvq_helpers import assert_attention_close, dev, host

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_call_twice():
    import torch
    from quantized_kv_cache_quant_gb300 import kvq

    b, hkv, hq, d, s = 4, 4, 32, 128, 32 * 50 + 77
    x = workloads.make_inputs(b, hkv, hq, d, s, 2, 123)
    cache = kvq.KiviCache(b, hkv, hq, d, 2, 2, 128, s + 2)
    cache.prefill(dev(x.k), dev(x.v))
    for step in range(2):                        # two calls in a row on the shared scratch array
        if step:
            cache.append(dev(x.k_new[step]), dev(x.v_new[step]))
        q = dev(x.q[step])
        ref = host(cache.decode(q)).astype(np.float64)
        out = torch.full((b, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        kvq.kv_decode_attention_noalloc(cache.desc, q, out, True, 0.0)
        assert_attention_close(host(out), ref)
    # fp16 output through the same call
    out16 = torch.empty((b, hq, d), dtype=torch.float16, device="cuda")
    kvq.kv_decode_attention_noalloc(cache.desc, q, out16, False, 0.0)
    assert_attention_close(host(out16).astype(np.float64), ref, fp16_out=True)


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
