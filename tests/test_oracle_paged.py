"""Pins of the paged, variable-length KIVI oracle against the contiguous one."""
import numpy as np
import pytest

from oracle import attention, kivi, layout, paged
from quantized_kv_cache_quant_gb300 import workloads


def _inputs(b, h, d, s, steps, seed):
    x = workloads.make_inputs(b, h, 2 * h, d, s + steps, max(steps, 1), seed)
    return x


@pytest.mark.parametrize("kb,vb,r", [(2, 2, 128), (4, 2, 64), (2, 4, 0)])
def test_identity_table_equal_lengths_is_the_contiguous_cache(kb, vb, r):
    b, h, d, s = 3, 2, 64, 32 * 6 + 50
    x = _inputs(b, h, d, s, 0, 5)
    k, v = x.k[:, :, :s], x.v[:, :, :s]
    c = kivi.KiviCache(b, h, d, kb, vb, r)
    c.prefill(k, v)
    ng = c.n_grouped // 32
    table = np.arange(b * 10, dtype=np.int32).reshape(b, 10)
    p = paged.PagedKiviCache(b, h, d, kb, vb, r, b * 10, table)
    p.prefill(k, v, [s] * b)
    packed = layout.pack_cache(c)
    pools = p.pools()
    for name, rec in packed.items():
        for bi in range(b):
            for g in range(ng):
                assert np.array_equal(pools[name][table[bi, g]], rec[bi, :, g]), (name, bi, g)
    q = x.q[0]
    sc = attention.default_scale(d)
    want = attention.decode_attention(q, c.keys_hat, c.values_hat, h, sc)
    got = attention.decode_attention(q, p.keys_hat, p.values_hat, h, sc)
    assert np.array_equal(got, want)


def test_each_sequence_is_its_own_cache_wherever_its_blocks_are():
    rng = np.random.default_rng(7)
    b, h, d = 4, 2, 128
    lens = [32 * 9 + 7, 129, 32 * 4, 31]
    x = _inputs(b, h, d, max(lens), 0, 9)
    table = rng.permutation(b * 12).astype(np.int32).reshape(b, 12)
    p = paged.PagedKiviCache(b, h, d, 2, 2, 128, b * 12, table)
    p.prefill(x.k, x.v, lens)
    pools = p.pools()
    used = set()
    for bi, n in enumerate(lens):
        one = kivi.KiviCache(1, h, d, 2, 2, 128)
        one.prefill(x.k[bi:bi + 1, :, :n], x.v[bi:bi + 1, :, :n])
        assert (p.n_grouped(bi), p.n_resid(bi)) == (one.n_grouped, one.n_resid)
        for name, rec in (layout.pack_cache(one).items() if one.n_grouped else ()):
            for g in range(rec.shape[2]):
                assert np.array_equal(pools[name][table[bi, g]], rec[0, :, g])
                used.add(int(table[bi, g]))
        kw, vw = p.window(bi)
        assert np.array_equal(kw, one.k_res[0]) and np.array_equal(vw, one.v_res[0])
    unused = [blk for blk in range(b * 12) if blk not in used]
    for name in pools:                                    # blocks no group uses stay empty
        assert not pools[name][unused].any()


def test_staggered_flushes_during_appends():
    b, h, d, r = 3, 2, 64, 64
    lens = [64 + 10, 64 + 63, 64 + 64]                    # grouped 32, 64, 64: windows 42, 63 and 64 (full)
    steps = 70
    x = _inputs(b, h, d, max(lens), steps, 11)
    table = np.arange(b * 8, dtype=np.int32).reshape(b, 8)
    p = paged.PagedKiviCache(b, h, d, 2, 2, r, b * 8, table)
    p.prefill(x.k, x.v, lens)
    assert [p.n_resid(i) for i in range(b)] == [42, 63, 64]
    flushed_at = {i: [] for i in range(b)}
    for t in range(steps):
        before = [p.n_grouped(i) for i in range(b)]
        p.append(x.k_new[t], x.v_new[t])
        for i in range(b):
            if p.n_grouped(i) != before[i]:
                flushed_at[i].append(t)
            assert p.n_grouped(i) + p.n_resid(i) == lens[i] + t + 1
    # a window flushes on the append that would overflow it (then refills from 1 to 64 tokens):
    # sequence 2 at once, 1 after one append, 0 after 22
    assert flushed_at == {0: [22], 1: [1, 65], 2: [0, 64]}


def test_pool_is_the_records_back_to_back():
    """One (block, kv head) entry of the pool is key codes, key meta, value
    codes, value meta in that order; the sizes add up to one group's records."""
    b, h, d = 2, 3, 64
    x = _inputs(b, h, d, 32 * 5 + 140, 0, 9)
    table = np.arange(b * 12, dtype=np.int32).reshape(b, 12)[:, ::-1].copy()
    p = paged.PagedKiviCache(b, h, d, 2, 4, 128, b * 12, table)
    p.prefill(x.k[:, :, :32 * 5 + 140], x.v[:, :, :32 * 5 + 140], [32 * 5 + 140, 40])
    pool, recs, off = p.pool(), p.pools(), p.record_offsets()
    nbytes = p.record_bytes()
    assert pool.shape == (b * 12, h, 32 * d * 2 // 8 + 4 * d + 32 * d * 4 // 8 + 128)
    assert off == {"k_codes": 0, "k_meta": 512, "v_codes": 768, "v_meta": 1792}
    for name in p.ORDER:
        assert np.array_equal(pool[:, :, off[name]:off[name] + nbytes[name]], recs[name])
