"""GPU parity of the KIVI path against the CPU oracle, through the C ABI.

Codes, scales and zero points must match bit for bit; attention must stay
within max-abs 2e-3 and relative L2 1e-3 of the float64 oracle computed on
the same dequantized values.
"""
import numpy as np
import pytest

from oracle import kivi
from oracle.attention import default_scale
from quantized_kv_cache_quant_gb300 import workloads

from kvq_helpers import (assert_all_grouped_bytes_equal, assert_attention_close, assert_grouped_bytes_equal,
                         assert_residual_equal, dev, host, oracle_attention, oracle_cache)

pytestmark = pytest.mark.gpu


def _kvq():
    from quantized_kv_cache_quant_gb300 import kvq
    return kvq


def _run(b, hkv, hq, d, s, kb=2, vb=2, r=128, steps=0, seed=0, max_tokens=None, out_fp32=True):
    kvq = _kvq()
    x = workloads.make_inputs(b, hkv, hq, d, s + steps, max(steps, 1), seed)
    k, v = x.k[:, :, :s], x.v[:, :, :s]
    mt = max_tokens or (s + steps + 1)
    gc = kvq.KiviCache(b, hkv, hq, d, kb, vb, r, mt)
    gc.prefill(dev(k), dev(v))
    oc = oracle_cache(dict(k_bits=kb, v_bits=vb, residual=r, max_tokens=mt), k, v)
    return kvq, x, gc, oc


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4), (2, 4), (4, 2)])
def test_prefill_bytes(d, kb, vb):
    kvq, x, gc, oc = _run(2, 3, 6, d, 32 * 7 + 128 + 5, kb, vb, seed=11)
    assert (gc.n_grouped, gc.n_resid) == (oc.n_grouped, oc.n_resid) == (256, 101)
    assert_grouped_bytes_equal(gc, oc)
    assert_residual_equal(gc, oc)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("gq", [1, 2, 3, 4, 5, 7, 8])
@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4), (2, 4)])
def test_decode_attention(d, gq, kb, vb):
    s = 32 * 37 + 128 - 9          # 37 groups (several splits), a ragged window
    kvq, x, gc, oc = _run(2, 2, 2 * gq, d, s, kb, vb, seed=100 + gq)
    q = x.q[0]
    out = host(gc.decode(dev(q)))
    ref = oracle_attention(oc, q, default_scale(d))
    assert_attention_close(out, ref)
    assert gc.status() == 0


def test_decode_fp16_output():
    kvq, x, gc, oc = _run(2, 2, 16, 128, 32 * 20 + 100, seed=7)
    q = x.q[0]
    out = host(gc.decode(dev(q), out_fp32=False)).astype(np.float64)
    ref = oracle_attention(oc, q, default_scale(128))
    assert_attention_close(out, ref, fp16_out=True)


@pytest.mark.parametrize("s", [1, 17, 100, 128])
def test_window_only(s):
    """S <= R: nothing is quantized; attention is exact fp16 attention."""
    kvq, x, gc, oc = _run(2, 2, 8, 64, s, seed=s)
    assert (gc.n_grouped, gc.n_resid) == (0, s)
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], default_scale(64)))


def test_fully_grouped_r0():
    """R = 0 with S a multiple of 32: every token lives in the grouped region."""
    kvq, x, gc, oc = _run(2, 4, 8, 128, 32 * 12, r=0, seed=3)
    assert (gc.n_grouped, gc.n_resid) == (384, 0)
    assert_grouped_bytes_equal(gc, oc)
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], default_scale(128)))


def test_zero_query_gives_mean_of_values():
    """q = 0: every score is 0, attention is the mean of the dequantized values."""
    kvq, x, gc, oc = _run(1, 2, 4, 128, 32 * 9 + 50, seed=17)
    q = np.zeros_like(x.q[0])
    out = host(gc.decode(dev(q)))
    for h in range(4):
        want = oc.values_hat(0, h // 2).mean(axis=0)
        assert np.allclose(out[0, h], want, atol=2e-3, rtol=0)


def test_fill_to_capacity_then_reject():
    """Append until the cache holds max_tokens; the next append is refused and
    the cache state is unchanged."""
    kvq = _kvq()
    x = workloads.make_inputs(1, 2, 2, 64, 100, 70, 8)
    gc = kvq.KiviCache(1, 2, 2, 64, 2, 2, 32, 170)
    oc = oracle_cache(dict(k_bits=2, v_bits=2, residual=32, max_tokens=170), x.k, x.v)
    gc.prefill(dev(x.k), dev(x.v))
    for step in range(70):
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
        oc.append(x.k_new[step], x.v_new[step])
    assert gc.n_grouped + gc.n_resid == 170
    with pytest.raises(kvq.KvqError) as e:
        gc.append(dev(x.k_new[0]), dev(x.v_new[0]))
    assert e.value.name == "KVQ_ERR_CAPACITY"
    assert gc.n_grouped + gc.n_resid == 170
    assert_grouped_bytes_equal(gc, oc)
    assert_residual_equal(gc, oc)
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], default_scale(64)))


def test_custom_softmax_scale():
    kvq, x, gc, oc = _run(1, 2, 4, 64, 300, seed=5)
    out = host(gc.decode(dev(x.q[0]), softmax_scale=0.05))
    assert_attention_close(out, oracle_attention(oc, x.q[0], np.float32(0.05)))


def test_tiny_workload_streaming():
    """The tiny workload: prefill 256 tokens (128 grouped + 128 fp16), 16 decode
    steps; the first step flushes the full window."""
    w = workloads.TINY
    kvq = _kvq()
    x = workloads.kivi_inputs(w)
    gc = kvq.KiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual, w.max_tokens)
    gc.prefill(dev(x.k), dev(x.v))
    oc = oracle_cache(dict(k_bits=2, v_bits=2, residual=128, max_tokens=w.max_tokens), x.k, x.v)
    assert (gc.n_grouped, gc.n_resid) == (128, 128)
    scale = default_scale(w.head_dim)
    for step in range(w.decode_steps):
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
        oc.append(x.k_new[step], x.v_new[step])
        assert (gc.n_grouped, gc.n_resid) == (oc.n_grouped, oc.n_resid)
        assert_grouped_bytes_equal(gc, oc)
        assert_residual_equal(gc, oc)
        out = host(gc.decode(dev(x.q[step])))
        assert_attention_close(out, oracle_attention(oc, x.q[step], scale))
    assert (gc.n_grouped, gc.n_resid) == (256, 16)


def test_r0_streaming_and_explicit_flush():
    kvq = _kvq()
    x = workloads.make_inputs(2, 2, 4, 64, 70, 40, 9)
    gc = kvq.KiviCache(2, 2, 4, 64, 2, 2, 0, 200)
    oc = oracle_cache(dict(k_bits=2, v_bits=2, residual=0, max_tokens=200), x.k, x.v)
    gc.prefill(dev(x.k), dev(x.v))
    assert (gc.n_grouped, gc.n_resid) == (64, 6)
    for step in range(40):
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
        oc.append(x.k_new[step], x.v_new[step])
        assert (gc.n_grouped, gc.n_resid) == (oc.n_grouped, oc.n_resid)
    assert_grouped_bytes_equal(gc, oc)
    assert_residual_equal(gc, oc)
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], default_scale(64)))


def test_explicit_flush_moves_the_remainder():
    kvq = _kvq()
    x = workloads.make_inputs(1, 2, 2, 128, 100, 1, 12)
    gc = kvq.KiviCache(1, 2, 2, 128, 2, 2, 128, 256)
    oc = oracle_cache(dict(k_bits=2, v_bits=2, residual=128, max_tokens=256), x.k, x.v)
    gc.prefill(dev(x.k), dev(x.v))
    assert (gc.n_grouped, gc.n_resid) == (0, 100)
    gc.flush()
    oc.flush()
    assert (gc.n_grouped, gc.n_resid) == (oc.n_grouped, oc.n_resid) == (96, 4)
    assert_grouped_bytes_equal(gc, oc)
    assert_residual_equal(gc, oc)
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], default_scale(128)))


def test_streaming_equals_prefill_on_device():
    """Prefill(S0) + n appends leaves the same bytes in every shared group as prefill(S0 + n)."""
    kvq = _kvq()
    x = workloads.make_inputs(2, 2, 4, 128, 256 + 200, 1, 13)
    a = kvq.KiviCache(2, 2, 4, 128, 2, 2, 128, 512)
    a.prefill(dev(x.k[:, :, :256]), dev(x.v[:, :, :256]))
    for t in range(256, 456):
        a.append(dev(x.k[:, :, t].copy()), dev(x.v[:, :, t].copy()))
    b = kvq.KiviCache(2, 2, 4, 128, 2, 2, 128, 512)
    b.prefill(dev(x.k), dev(x.v))
    n = min(a.n_grouped, b.n_grouped) // 32
    for name in ("k_codes", "k_meta", "v_codes", "v_meta"):
        assert np.array_equal(host(a.grouped_view(name))[:, :, :n], host(b.grouped_view(name))[:, :, :n]), name


# ---------------------------------------------------------------------------
# full-size workloads: all bytes (or every flushed group) and sampled heads
# ---------------------------------------------------------------------------

def _sample_heads(b, hq, n, seed):
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (b - 1, hq - 1)}
    while len(picks) < n:
        picks.add((int(rng.integers(b)), int(rng.integers(hq))))
    return sorted(picks)


def test_decode_more_pairs_than_resident_blocks():
    """1024 (batch row, kv head) pairs, more than the GPU keeps resident: the
    grid is the stream-K cut, whose blocks each cover two or three pairs (one
    partial per pair) with odd group counts per segment."""
    b, hkv, gq, d = 64, 16, 2, 64
    s = 32 * 37 + 128 - 9                      # 37 groups + 119 window tokens per pair
    kvq, x, gc, oc = _run(b, hkv, hkv * gq, d, s, seed=21)
    heads = _sample_heads(b, hkv * gq, 48, 21)
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], default_scale(d), heads), heads)
    assert gc.status() == 0


@pytest.mark.parametrize("n_resid", [32, 33, 64, 65, 96, 127])
def test_decode_window_chunk_edges(n_resid):
    """Window fills at and around the 32-token chunk boundaries, after a flush,
    with grouped tokens in front."""
    b, hkv, hq, d = 2, 3, 12, 128
    s = 32 * 9 + 128                           # 9 groups + a full window
    kvq, x, gc, oc = _run(b, hkv, hq, d, s, steps=n_resid, seed=31 + n_resid)
    for step in range(n_resid):                # the first append flushes the full window
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
        oc.append(x.k_new[step], x.v_new[step])
    assert (gc.n_grouped, gc.n_resid) == (oc.n_grouped, oc.n_resid) == (32 * 13, n_resid)
    q = x.q[n_resid - 1]
    out = host(gc.decode(dev(q)))
    assert_attention_close(out, oracle_attention(oc, q, default_scale(d)))
    assert gc.status() == 0


@pytest.mark.parametrize("w", [workloads.MHA_4K, workloads.GQA_8K_2BIT, workloads.GQA_8K_4BIT], ids=lambda w: w.name)
def test_full_size_decode(w):
    kvq = _kvq()
    x = workloads.kivi_inputs(w)
    gc = kvq.KiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual, w.max_tokens)
    gc.prefill(dev(x.k), dev(x.v))
    oc = oracle_cache(dict(k_bits=w.k_bits, v_bits=w.v_bits, residual=w.residual, max_tokens=w.max_tokens), x.k, x.v)
    assert_all_grouped_bytes_equal(gc, oc, rows_per_chunk=4)
    assert_residual_equal(gc, oc)
    scale = default_scale(w.head_dim)
    # attention on every query head over the prefilled cache, then one streaming decode step
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], scale))
    gc.append(dev(x.k_new[0]), dev(x.v_new[0]))
    oc.append(x.k_new[0], x.v_new[0])
    assert_grouped_bytes_equal(gc, oc, groups=list(range(oc.n_grouped // 32 - 4, oc.n_grouped // 32)))
    out = host(gc.decode(dev(x.q[0])))
    assert_attention_close(out, oracle_attention(oc, x.q[0], scale))
    assert gc.status() == 0


def test_full_size_streaming_128k():
    """128K streaming workload: prefill 131072 tokens (every byte of all 4092
    groups x 32 pairs compared), 512 decode steps with a flush every 128
    steps; every flushed group is compared bit for bit, attention is checked
    on every query head at steps 0 and 511 and on sampled heads at steps 1,
    127, 128, 255 and 256."""
    w = workloads.STREAM_128K
    kvq = _kvq()
    x = workloads.kivi_inputs(w)
    gc = kvq.KiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual, w.max_tokens)
    gc.prefill(dev(x.k), dev(x.v))
    oc = oracle_cache(dict(k_bits=2, v_bits=2, residual=128, max_tokens=w.max_tokens), x.k, x.v)
    assert (gc.n_grouped, gc.n_resid) == (130944, 128)
    assert_all_grouped_bytes_equal(gc, oc)
    heads = _sample_heads(w.batch, w.q_heads, 24, w.seed)
    every = {0, w.decode_steps - 1}
    scale = default_scale(w.head_dim)
    check = {0, 1, 127, 128, 255, 256, 511}
    for step in range(w.decode_steps):
        before = gc.n_grouped
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
        oc.append(x.k_new[step], x.v_new[step])
        if gc.n_grouped != before:
            ng = gc.n_grouped // 32
            assert_grouped_bytes_equal(gc, oc, groups=list(range(ng - 4, ng)))
        out = gc.decode(dev(x.q[step]))
        if step in every:
            assert_attention_close(host(out), oracle_attention(oc, x.q[step], scale))
        elif step in check:
            assert_attention_close(host(out), oracle_attention(oc, x.q[step], scale, heads), heads)
    assert (gc.n_grouped, gc.n_resid) == (131456, 128)
    assert_residual_equal(gc, oc)
    assert gc.status() == 0


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4)])
def test_prefill_exact_ties(kb, vb):
    """Quotients that land exactly on half-integers (ties, rounded to even) and
    just beside them: every code must match the oracle's IEEE fp32 formula."""
    kvq = _kvq()
    rng = np.random.default_rng(kb * 10 + vb)
    b, h, d, s = 2, 2, 128, 32 * 8
    levels = 2 ** kb - 1
    k = np.empty((b, h, s, d), np.float16)
    for g in range(s // 32):
        step = np.float16(2.0 ** int(rng.integers(-6, 3)))
        base = np.float16(int(rng.integers(-20, 20)) * float(step))
        half = rng.integers(0, 2 * levels + 1, size=(b, h, 32, d))          # multiples of step / 2
        half[:, :, 0, :], half[:, :, 1, :] = 0, 2 * levels                   # fix min and max
        k[:, :, 32 * g:32 * g + 32] = (np.float64(base) + half * float(step) / 2).astype(np.float16)
    nudge = rng.random(k.shape) < 0.2                                       # some values one ulp off a tie
    k = np.where(nudge, np.nextafter(k, np.float16(np.inf)), k).astype(np.float16)
    v = k.copy()
    gc = kvq.KiviCache(b, h, 2 * h, d, kb, vb, 0, s)
    gc.prefill(dev(k), dev(v))
    oc = oracle_cache(dict(k_bits=kb, v_bits=vb, residual=0, max_tokens=s), k, v)
    assert_grouped_bytes_equal(gc, oc)


def _f16_range(mn, mx):
    """Every fp16 value in [mn, mx] in increasing order (-0 left out)."""
    def key(h):
        b = int(np.array([h], np.float16).view(np.uint16)[0])
        return -(b & 0x7FFF) if b & 0x8000 else b
    ks = np.arange(key(mn), key(mx) + 1)
    bits = np.where(ks >= 0, ks, 0x8000 | (-ks)).astype(np.uint16)
    return bits.view(np.float16)


def _code_steps(mn, mx, bits):
    """The fp16 values where the oracle's code changes for a group of min mn and
    max mx, and the values just below them: rows [mn, mx, x] keep the group's
    min and max, so their third code is code(x)."""
    xs = _f16_range(mn, mx)
    rows = np.stack([np.full(xs.size, mn, np.float16), np.full(xs.size, mx, np.float16), xs], axis=-1)
    codes = kivi.quantize_groups(rows, bits)[0][:, 2].astype(int)
    up = np.nonzero(np.diff(codes) > 0)[0]
    return np.unique(np.concatenate([xs[up], xs[up + 1]]))


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4), (2, 4)])
def test_prefill_at_every_code_step(kb, vb):
    """Groups whose elements sit on both sides of every step of the code
    function (found by the oracle over all fp16 values of the group's range),
    for ranges that are symmetric about 0 (a step near 0, where fp32 rounding of
    x - min moves it), tiny (subnormal scales), up to +-65504, one-signed,
    constant and zero: every byte must match."""
    kvq = _kvq()
    rng = np.random.default_rng(kb * 10 + vb + 7)
    ranges = [(-3.0, 3.0), (-1000.0, 1000.0), (-65504.0, 65504.0), (-1e-6, 1e-6), (-6e-8, 6e-8), (0.0, 2.0),
              (-2.0, 0.0), (1.0, 1.0), (0.0, 0.0), (-5e4, 3e-5), (-3e-5, 5e4), (-1000.0, 1e-3), (100.0, 100.5),
              (-60000.0, 2.0), (-0.75, 0.25), (5e-5, 7e-5)]
    for _ in range(16):
        a, c = sorted(rng.standard_normal(2) * 10.0 ** rng.uniform(-6, 4.5))
        ranges.append((a, c))
    groups = []
    for a, c in ranges:
        mn, mx = np.float16(a), np.float16(c)
        steps = _code_steps(mn, mx, max(kb, vb))
        steps = steps if kb == vb else np.unique(np.concatenate([steps, _code_steps(mn, mx, min(kb, vb))]))
        groups.append((mn, mx, steps))
    b, h, d, ng = 2, 2, 128, 4
    s = 32 * ng
    k = np.empty((b, h, s, d), np.float16)
    v = np.empty((b, h, s, d), np.float16)
    for bi in range(b):
        for hi in range(h):
            for g in range(ng):
                for ch in range(d):                    # key group: channel ch over 32 tokens
                    mn, mx, steps = groups[int(rng.integers(len(groups)))]
                    col = rng.choice(_f16_range(mn, mx), 30)
                    take = steps[:30] if steps.size <= 30 else rng.choice(steps, 30, replace=False)
                    col[:take.size] = take
                    k[bi, hi, 32 * g:32 * g + 32, ch] = rng.permutation(np.concatenate([[mn, mx], col]))
                for t in range(32 * g, 32 * g + 32):   # value group: token t over 128 channels
                    mn, mx, steps = groups[int(rng.integers(len(groups)))]
                    row = rng.choice(_f16_range(mn, mx), d - 2)
                    row[:steps.size] = steps[:d - 2]
                    v[bi, hi, t] = rng.permutation(np.concatenate([[mn, mx], row]))
    gc = kvq.KiviCache(b, h, 2 * h, d, kb, vb, 0, s)
    gc.prefill(dev(k), dev(v))
    oc = oracle_cache(dict(k_bits=kb, v_bits=vb, residual=0, max_tokens=s), k, v)
    assert_grouped_bytes_equal(gc, oc)
