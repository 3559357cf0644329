"""Magnitude edge cases of KIVI decode attention, for both decode kernels
(query heads per kv head above 4: heads on the tile rows; at most 4: the
swapped-operand kernel) and for the contiguous and the paged cache:

* tiny: keys and values scaled by 2^-16, so most group scales are fp16
  subnormals (below 2^-14) and every product p * s_t of the value path lies
  below fp16's normal range;
* fp16_max: keys and values whose group ranges reach +-65000, so the key
  and value scales sit near (65000 + 65000) / 3, where the bound
  2^0.5 * s_t < 65504 of the value operand is tight;
* dominant: one token per (batch row, kv head) whose key points along its
  query heads with a logit far above the rest, and whose values are tiny
  (an attention-sink-like token); it lies in the grouped region for some
  pairs and in the fp16 window for the others.

The FP8 and NVFP4 paged decodes take the first two at the same magnitudes.

Attention is linear in the values, so outputs are compared after dividing by
the values' magnitude M (the same bars as the other parity tests: max-abs
2e-3 and relative L2 1e-3 of the float64 oracle on the same dequantized
values, read relative to M).
"""
import numpy as np
import pytest

from oracle import attention, kivi, paged
from oracle.attention import default_scale
from quantized_kv_cache_quant_gb300 import workloads

from kvq_helpers import assert_attention_close, dev, host, oracle_attention, oracle_cache

pytestmark = pytest.mark.gpu

TINY = 2.0 ** -16
BIG = 65000.0


def _edge_inputs(kind, b, hkv, hq, d, s, seed, windows=None):
    """fp16 k, v [B, Hkv, S, D], q [B, Hq, D] and the value magnitude M.
    windows[b] (paged): the first token of sequence b's window, so that the
    dominant token can be placed there."""
    x = workloads.make_inputs(b, hkv, hq, d, s, 1, seed)
    k = x.k.astype(np.float64)
    v = x.v.astype(np.float64)
    q = x.q[0].astype(np.float64)
    rng = np.random.default_rng(seed + 7)
    if kind == "tiny":
        k *= TINY
        v *= TINY
        q *= 64.0
        m = TINY
    elif kind == "fp16_max":
        # in every 32-token group channel c reaches +BIG at token c % 32 and -BIG at (c + 16) % 32
        k = k / np.abs(k).max() * BIG
        c = np.arange(d)
        for g0 in range(0, s - 31, 32):
            k[:, :, g0 + c % 32, c] = BIG
            k[:, :, g0 + (c + 16) % 32, c] = -BIG
        # every token spans [-BIG, +BIG] across its channels
        v = v / np.abs(v).max(axis=-1, keepdims=True) * BIG
        v[..., 0] = BIG
        v[..., 1] = -BIG
        q *= 2.0 ** -12
        m = BIG
    elif kind == "dominant":
        gq = hq // hkv
        m = TINY
        v *= TINY
        first_window = windows if windows is not None else [kivi.prefill_split(s, 128)[0]] * b
        for bi in range(b):
            for h in range(hkv):
                qs = q[bi, h * gq:(h + 1) * gq]
                u = qs.sum(axis=0)
                u /= np.linalg.norm(u)
                # the rest's largest logit (on the unquantized keys), then a margin of 30
                rest = (qs @ k[bi, h].T).max() / np.sqrt(d)
                own = (qs @ u).min() / np.sqrt(d)
                assert own > 0.05
                alpha = (rest + 30.0) / own
                if (bi + h) % 2 == 1:                  # in the fp16 window
                    t = first_window[bi] + int(rng.integers(0, 8))
                else:                                  # in one of the first four groups
                    t = int(rng.integers(0, 32 * 4))
                k[bi, h, t] = alpha * u
    else:
        raise ValueError(kind)
    return k.astype(np.float16), v.astype(np.float16), q.astype(np.float16), m


def _check_kind(kind, oc, kb, vb):
    """The inputs really are at the edge the test names."""
    if kind == "tiny":
        ks = oc.k_scale.astype(np.float64)
        vs = oc.v_scale.astype(np.float64)
        assert np.mean((ks > 0) & (ks < 2.0 ** -14)) > 0.5
        assert np.mean((vs > 0) & (vs < 2.0 ** -14)) > 0.9
    elif kind == "fp16_max":
        # group ranges of about 2 * BIG: scales near 2 * BIG / (2^bits - 1)
        assert oc.k_scale.astype(np.float64).max() >= 0.99 * 2 * BIG / (2 ** kb - 1)
        assert oc.v_scale.astype(np.float64).max() >= 0.99 * 2 * BIG / (2 ** vb - 1)


KINDS = ["tiny", "fp16_max", "dominant"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("gq,d,kb,vb", [(8, 128, 2, 2), (4, 128, 2, 2), (1, 64, 2, 2), (8, 128, 4, 4),
                                        (2, 128, 4, 2)])
def test_contiguous_edges(kind, gq, d, kb, vb):
    from quantized_kv_cache_quant_gb300 import kvq
    b, hkv = 2, 2
    hq = hkv * gq
    s = 32 * 40 + 77                                   # 40 groups + 77 window tokens after the prefill split
    k, v, q, m = _edge_inputs(kind, b, hkv, hq, d, s, 100 + gq + d + kb)
    gc = kvq.KiviCache(b, hkv, hq, d, kb, vb, 128, s)
    gc.prefill(dev(k), dev(v))
    oc = oracle_cache(dict(k_bits=kb, v_bits=vb, residual=128, max_tokens=s), k, v)
    _check_kind(kind, oc, kb, vb)
    ref = oracle_attention(oc, q, default_scale(d))
    out = host(gc.decode(dev(q)))
    assert_attention_close(out / m, ref / m)
    assert gc.status() == 0


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("gq,kb,vb", [(8, 2, 2), (2, 2, 2), (4, 4, 4)])
def test_paged_edges(kind, gq, kb, vb):
    from quantized_kv_cache_quant_gb300 import kvq
    hkv, d, r = 2, 128, 128
    lens = [32 * 30 + 50, 32 * 5 + 128, 32 * 12 + 1]
    b = len(lens)
    hq = hkv * gq
    s = max(lens)
    windows = [kivi.prefill_split(n, r)[0] for n in lens]
    k, v, q, m = _edge_inputs(kind, b, hkv, hq, d, s, 200 + gq + kb, windows=windows)
    if kind == "dominant":
        # a dominant token past a sequence's length would not be seen: keep every one inside
        for bi, n in enumerate(lens):
            assert windows[bi] + 8 <= n
    gcap = -(-s // 32)
    nb = b * gcap
    table = workloads.block_table(b, gcap, 5)
    gc = kvq.PagedKiviCache(b, hkv, hq, d, kb, vb, r, s, nb)
    gc.table.copy_(dev(table))
    gc.prefill(dev(k), dev(v), lens)
    oc = paged.PagedKiviCache(b, hkv, d, kb, vb, r, nb, table)
    oc.prefill(k, v, lens)
    ref = attention.decode_attention(q, oc.keys_hat, oc.values_hat, oc.H, default_scale(d))
    out = host(gc.decode(dev(q)))
    assert_attention_close(out / m, ref / m)


# ---------------------------------------------------------------------------
# The FP8 and NVFP4 paged decodes at the same magnitudes: keys and values
# scaled by 2^-16 (the tensor scales shrink with them) and up to +-65000.
# ---------------------------------------------------------------------------
def _scaled(kind, x):
    k, v, q = x.k.astype(np.float64), x.v.astype(np.float64), x.q[0].astype(np.float64)
    if kind == "tiny":
        k, v, q, m = k * TINY, v * TINY, q * 64.0, TINY
    else:
        k = k / np.abs(k).max() * BIG
        v = v / np.abs(v).max() * BIG
        q, m = q * 2.0 ** -12, BIG
    return k.astype(np.float16), v.astype(np.float16), q.astype(np.float16), m


@pytest.mark.parametrize("kind", ["tiny", "fp16_max"])
@pytest.mark.parametrize("gq", [4, 1])
def test_fp8_decode_edges(kind, gq):
    from oracle import fp8
    from test_gpu_fp8 import KEY, VALUE, _decode, _oracle_decode, _quantize
    b, hkv, d, s = 2, 2, 128, 16 * 40 + 5
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 300 + gq)
    k, v, q, m = _scaled(kind, x)
    nb = -(-s // 16)
    table = workloads.block_table(b, nb, 7)
    kp, ks = _quantize(k, table, b * nb, KEY)
    vp, vs = _quantize(v, table, b * nb, VALUE)
    lens = np.array([s, 16 * 9 + 3])
    out, status = _decode(q, kp, vp, ks, vs, table, lens, hkv, b * nb, s)
    assert status == 0
    ref = _oracle_decode(q, k, v, fp8.dynamic_scale(k), fp8.dynamic_scale(v), lens)
    assert_attention_close(out / m, ref / m)


@pytest.mark.parametrize("kind", ["tiny", "fp16_max"])
@pytest.mark.parametrize("gq", [8, 4, 1])
def test_nvfp4_decode_edges(kind, gq):
    from test_gpu_nvfp4 import _decode, _oracle_decode
    b, hkv, d, s = 2, 2, 128, 16 * 40 + 5
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 400 + gq)
    k, v, q, m = _scaled(kind, x)
    xs = workloads.KVInputs(k, v, q[None], x.k_new, x.v_new)
    nb = -(-s // 16)
    table = workloads.block_table(b, nb, 9)
    lens = np.array([s, 16 * 9 + 3], np.int32)
    got = _decode(xs, table, nb, lens, hkv * gq)
    assert_attention_close(got / m, _oracle_decode(xs, lens) / m)
