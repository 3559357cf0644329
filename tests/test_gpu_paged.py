"""GPU parity of the paged, variable-length KIVI cache against the paged oracle,
through the C ABI.

Pool blocks (for every group a sequence holds), windows and per-sequence state
must match bit for bit; attention must stay within the bars of the contiguous
path (max-abs 2e-3, relative L2 1e-3 of the float64 oracle on the same
dequantized values).
"""
import numpy as np
import pytest

from oracle import attention, kivi, layout, paged
from oracle.attention import default_scale
from quantized_kv_cache_quant_gb300 import workloads

from kvq_helpers import assert_attention_close, dev, host

pytestmark = pytest.mark.gpu

NAMES = ("k_codes", "k_meta", "v_codes", "v_meta")


def _kvq():
    from quantized_kv_cache_quant_gb300 import kvq
    return kvq


def _build(lens, hkv=2, hq=4, d=64, kb=2, vb=2, r=128, steps=0, seed=0, permute=True, extra=0):
    """A GPU paged cache and the paged oracle, both prefilled with the same
    inputs (sequence b uses its first lens[b] tokens)."""
    kvq = _kvq()
    b = len(lens)
    s = max(max(lens), 1)
    x = workloads.make_inputs(b, hkv, hq, d, s, max(steps, 1), seed)
    max_tokens = s + steps + extra
    gcap = -(-max_tokens // 32)
    nb = b * gcap
    table = (workloads.block_table(b, gcap, seed + 1) if permute
             else np.arange(nb, dtype=np.int32).reshape(b, gcap))
    gc = kvq.PagedKiviCache(b, hkv, hq, d, kb, vb, r, max_tokens, nb)
    gc.table.copy_(dev(table))
    gc.buffers["pool"].fill_(0xA5)        # a sentinel: blocks no group uses keep it
    gc.prefill(dev(x.k), dev(x.v), lens)
    oc = paged.PagedKiviCache(b, hkv, d, kb, vb, r, nb, table)
    oc.prefill(x.k, x.v, lens)
    return kvq, x, gc, oc, table


def _assert_state(gc, oc):
    for b in range(oc.B):
        assert (gc.n_grouped(b), gc.n_resid(b)) == (oc.n_grouped(b), oc.n_resid(b)), b


def _assert_pools_equal(gc, oc, table):
    """Every block a group uses holds the oracle's pool entries (the four
    records back to back); every other block still holds the sentinel."""
    want = oc.pool()
    used = np.zeros(oc.num_blocks, bool)
    for b in range(oc.B):
        used[table[b, :oc.n_grouped(b) // 32]] = True
    got = host(gc.pool_view())
    assert got.shape == want.shape
    if not np.array_equal(got[used], want[used]):
        bad = np.argwhere(got[used] != want[used])
        raise AssertionError(f"{len(bad)} bytes differ, first at {bad[:5].tolist()}")
    assert np.all(got[~used] == 0xA5)


def _assert_windows_equal(gc, oc):
    for b in range(oc.B):
        n = oc.n_resid(b)
        kw, vw = oc.window(b)
        for name, want in (("k_res", kw), ("v_res", vw)):
            got = host(gc.residual_view(name))[b, :, :n]
            assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), (name, b)


def _oracle_out(oc, q, scale, heads=None):
    return attention.decode_attention(q, oc.keys_hat, oc.values_hat, oc.H, scale, heads)


# ragged lengths: empty, window-only, exactly R, one past R, several groups plus a ragged window
LENS = [0, 1, 100, 128, 129, 161, 32 * 20 + 77, 32 * 9]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4), (2, 4), (4, 2)])
def test_prefill_pools_windows_state(d, kb, vb):
    kvq, x, gc, oc, table = _build(LENS, d=d, kb=kb, vb=vb, seed=21)
    _assert_state(gc, oc)
    _assert_pools_equal(gc, oc, table)
    _assert_windows_equal(gc, oc)


@pytest.mark.parametrize("r", [0, 32, 64])
def test_prefill_other_windows(r):
    kvq, x, gc, oc, table = _build(LENS, d=128, r=r, seed=22 + r)
    _assert_state(gc, oc)
    _assert_pools_equal(gc, oc, table)
    _assert_windows_equal(gc, oc)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("gq", [1, 4, 5, 8])
@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4), (2, 4)])
def test_decode_attention(d, gq, kb, vb):
    lens = [1, 100, 129, 32 * 37 + 128 - 9, 32 * 5, 161, 32 * 61 + 3]
    kvq, x, gc, oc, table = _build(lens, hkv=2, hq=2 * gq, d=d, kb=kb, vb=vb, seed=30 + gq)
    q = x.q[0]
    out = host(gc.decode(dev(q)))
    assert_attention_close(out, _oracle_out(oc, q, default_scale(d)))
    assert gc.status() == 0


def test_decode_fp16_output_and_custom_scale():
    kvq, x, gc, oc, table = _build([700, 33, 1500], hkv=2, hq=16, d=128, seed=40)
    q = x.q[0]
    out = host(gc.decode(dev(q), out_fp32=False)).astype(np.float64)
    assert_attention_close(out, _oracle_out(oc, q, default_scale(128)), fp16_out=True)
    out = host(gc.decode(dev(q), softmax_scale=0.05))
    assert_attention_close(out, _oracle_out(oc, q, np.float32(0.05)))


def test_decode_rejects_an_empty_sequence():
    kvq, x, gc, oc, table = _build([0, 50], seed=41)
    with pytest.raises(kvq.KvqError) as e:
        gc.decode(dev(x.q[0]))
    assert e.value.name == "KVQ_ERR_ARG"


@pytest.mark.parametrize("r", [128, 0])
def test_streaming_flushes_at_each_sequence_own_time(r):
    """Appends cross window flushes at different steps for each sequence; bytes,
    windows and state follow the oracle after every step, attention at a few."""
    lens = [0, 5, 127, 128, 200, 32 * 4 + 31, 31]
    steps = 70
    kvq, x, gc, oc, table = _build(lens, hkv=2, hq=8, d=64, r=r, steps=steps, seed=50 + r)
    for step in range(steps):
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
        oc.append(x.k_new[step], x.v_new[step])
        _assert_state(gc, oc)
        if step % 23 == 0 or step == steps - 1:
            _assert_pools_equal(gc, oc, table)
            _assert_windows_equal(gc, oc)
            q = x.q[step]
            assert_attention_close(host(gc.decode(dev(q))), _oracle_out(oc, q, default_scale(64)))
    assert gc.status() == 0


def test_explicit_flush():
    kvq, x, gc, oc, table = _build([3, 20, 100, 128, 32 * 3 + 90], d=128, seed=60)
    gc.flush()
    for c in oc.seqs:
        c.flush()
    _assert_state(gc, oc)
    _assert_pools_equal(gc, oc, table)
    _assert_windows_equal(gc, oc)
    gc.flush()                      # nothing left to flush: no change
    _assert_state(gc, oc)
    q = x.q[0]
    assert_attention_close(host(gc.decode(dev(q))), _oracle_out(oc, q, default_scale(128)))


def test_identity_table_equal_lengths_matches_the_contiguous_cache():
    """Same inputs, same lengths: the paged pools hold exactly the contiguous
    cache's grouped records, and both decodes agree with the oracle."""
    kvq = _kvq()
    b, hkv, hq, d, s = 3, 2, 8, 128, 32 * 30 + 70
    kvq_, x, gc, oc, table = _build([s] * b, hkv=hkv, hq=hq, d=d, seed=70, permute=False)
    cc = kvq.KiviCache(b, hkv, hq, d, 2, 2, 128, s)
    cc.prefill(dev(x.k[:, :, :s]), dev(x.v[:, :, :s]))
    ng = cc.n_grouped // 32
    for name in NAMES:
        got = host(gc.pool_view(name))[table[:, :ng].reshape(-1)].reshape(b, ng, hkv, -1).transpose(0, 2, 1, 3)
        assert np.array_equal(got, host(cc.grouped_view(name))[:, :, :ng]), name
    q = x.q[0]
    ref = _oracle_out(oc, q, default_scale(d))
    assert_attention_close(host(gc.decode(dev(q))), ref)
    assert_attention_close(host(cc.decode(dev(q))), ref)


def test_out_of_range_table_entries():
    """A quantize skips groups whose entry is outside [0, num_blocks) (the pool
    keeps its sentinel); the decode clamps such entries into the pool and still
    completes with finite outputs."""
    kvq, x, gc, oc, table = _build([32 * 8 + 128], d=64, seed=80)
    bad = table.copy()
    bad[0, 2] = -1
    bad[0, 5] = gc.pcfg.num_blocks
    gc.table.copy_(dev(bad))
    gc.buffers["pool"].fill_(0xA5)
    gc.prefill(dev(x.k), dev(x.v), [32 * 8 + 128])
    want = oc.pools()
    for name in NAMES:
        got = host(gc.pool_view(name))
        for g in range(8):
            if g in (2, 5):
                continue
            assert np.array_equal(got[bad[0, g]], want[name][table[0, g]]), (name, g)
        untouched = np.setdiff1d(np.arange(gc.pcfg.num_blocks), bad[0, [0, 1, 3, 4, 6, 7]])
        assert np.all(got[untouched] == 0xA5), name
    out = host(gc.decode(dev(x.q[0])))
    assert np.all(np.isfinite(out))
    assert gc.status() == 0


def test_most_sequences():
    """KVQ_PAGED_MAX_SEQS sequences of short, ragged lengths: the per-sequence
    ranges of every launch at their largest."""
    kvq = _kvq()
    rng = np.random.default_rng(90)
    lens = rng.integers(1, 300, size=kvq.PAGED_MAX_SEQS).tolist()
    kvq_, x, gc, oc, table = _build(lens, hkv=1, hq=2, d=64, steps=3, seed=90)
    for step in range(3):
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
        oc.append(x.k_new[step], x.v_new[step])
    _assert_state(gc, oc)
    _assert_pools_equal(gc, oc, table)
    _assert_windows_equal(gc, oc)
    q = x.q[2]
    assert_attention_close(host(gc.decode(dev(q))), _oracle_out(oc, q, default_scale(64)))


def _sampled_sequence_oracle(w, x, lens, b):
    """The contiguous oracle of sequence b alone (its own KIVI cache)."""
    c = kivi.KiviCache(1, w.kv_heads, w.head_dim, w.k_bits, w.v_bits, w.residual)
    c.prefill(x.k[b:b + 1, :, :lens[b]], x.v[b:b + 1, :, :lens[b]])
    return c


@pytest.mark.parametrize("w", [workloads.PAGED_VAR_16K, workloads.PAGED_GQA_8K], ids=lambda w: w.name)
def test_full_size_sampled(w):
    """The table workloads at full size, launched as the table times them:
    the records and attention of three sampled sequences against their own
    oracle caches, the state of all."""
    kvq = _kvq()
    x, lens, table = workloads.paged_inputs(w, steps=1)
    gc = kvq.PagedKiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual,
                            w.max_tokens, w.num_blocks)
    gc.table.copy_(dev(table))
    gc.prefill(dev(x.k), dev(x.v), lens.tolist())
    q = x.q[0]
    out = host(gc.decode(dev(q)))
    assert gc.status() == 0
    gq = w.q_heads // w.kv_heads
    rng = np.random.default_rng(w.seed)
    for b in sorted(rng.choice(w.batch, size=3, replace=False).tolist()):
        c = _sampled_sequence_oracle(w, x, lens, b)
        assert (gc.n_grouped(b), gc.n_resid(b)) == (c.n_grouped, c.n_resid)
        ng = c.n_grouped // 32
        packed = layout.pack_cache(c)
        for name in NAMES:
            got = host(gc.pool_view(name))[table[b, :ng]]            # [ng, H, bytes]
            assert np.array_equal(got.transpose(1, 0, 2), packed[name][0]), (name, b)
        heads = rng.choice(w.q_heads, size=6, replace=False)
        for hq in heads:
            h = hq // gq
            ref = attention.softmax_attend(q[b, hq], c.keys_hat(0, h), c.values_hat(0, h), default_scale(w.head_dim))
            got = out[b, hq].astype(np.float64)
            assert np.max(np.abs(got - ref)) <= 2e-3, (b, hq)
            assert np.linalg.norm(got - ref) <= 1e-3 * np.linalg.norm(ref), (b, hq)


def test_full_size_streaming_sampled():
    """The mixed-length table workload streamed for 130 decode steps: every
    sequence flushes its window once at its own step; state of all sequences,
    records and windows of three sampled sequences against their own oracle
    caches, and attention of their heads at the last step."""
    kvq = _kvq()
    w = workloads.PAGED_VAR_16K
    steps = 130
    x, lens, table = workloads.paged_inputs(w, steps=steps)
    gc = kvq.PagedKiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual,
                            w.max_len + steps, w.batch * (-(-(w.max_len + steps) // 32)))
    table = workloads.block_table(w.batch, gc.desc.groups_cap, w.seed + 1000)
    gc.table.copy_(dev(table))
    gc.prefill(dev(x.k), dev(x.v), lens.tolist())
    for step in range(steps):
        gc.append(dev(x.k_new[step]), dev(x.v_new[step]))
    q = x.q[steps - 1]
    out = host(gc.decode(dev(q)))
    assert gc.status() == 0
    gq = w.q_heads // w.kv_heads
    rng = np.random.default_rng(w.seed + 1)
    for b in sorted(rng.choice(w.batch, size=3, replace=False).tolist()):
        c = _sampled_sequence_oracle(w, x, lens, b)
        for step in range(steps):
            c.append(x.k_new[step][b:b + 1], x.v_new[step][b:b + 1])
        assert (gc.n_grouped(b), gc.n_resid(b)) == (c.n_grouped, c.n_resid), b
        ng = c.n_grouped // 32
        packed = layout.pack_cache(c)
        for name in NAMES:
            got = host(gc.pool_view(name))[table[b, :ng]]
            assert np.array_equal(got.transpose(1, 0, 2), packed[name][0]), (name, b)
        for name, want in (("k_res", c.k_res[0]), ("v_res", c.v_res[0])):
            got = host(gc.residual_view(name))[b, :, :c.n_resid]
            assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), (name, b)
        for hq in rng.choice(w.q_heads, size=4, replace=False):
            h = hq // gq
            ref = attention.softmax_attend(q[b, hq], c.keys_hat(0, h), c.values_hat(0, h), default_scale(w.head_dim))
            got = out[b, hq].astype(np.float64)
            assert np.max(np.abs(got - ref)) <= 2e-3, (b, hq)
            assert np.linalg.norm(got - ref) <= 1e-3 * np.linalg.norm(ref), (b, hq)
