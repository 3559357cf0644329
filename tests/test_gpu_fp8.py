"""GPU parity of the FP8 E4M3 paged path against the CPU oracle, through the C ABI.

FP8 bytes and the per-tensor scale must match bit for bit; attention must stay
within max-abs 2e-3 and relative L2 1e-3 of the float64 oracle computed on the
same dequantized values.
"""
import numpy as np
import pytest

from oracle import attention, fp8, layout
from oracle.attention import default_scale
from quantized_kv_cache_quant_gb300 import workloads

from kvq_helpers import assert_attention_close, dev, host

pytestmark = pytest.mark.gpu


def _kvq():
    from quantized_kv_cache_quant_gb300 import kvq
    return kvq


# the oracle's in-block order of each role: keys in the m16n8k32 order (layout id 2), values 1
KEY, VALUE = 2, 1


def _quantize(x16, table, num_blocks, vl, static_scale=None, fmt="e4m3", per_head=False):
    """A key (vl = KEY) or value (vl = VALUE) pool; static_scale: None (dynamic), a
    scalar, or per head an array [H]. Returns (pool, its scale tensor)."""
    import torch
    kvq = _kvq()
    b, h, s, d = x16.shape
    p = kvq.Fp8Pool(kvq.ROLE_KEY if vl == KEY else kvq.ROLE_VALUE, num_blocks, h, d,
                    fp8_format=kvq.FP8_FORMATS[fmt], per_head=per_head)
    p.buf.fill_(0xAB)
    n = h if per_head else 1
    init = np.full(n, -1.0, np.float32) if static_scale is None else np.broadcast_to(
        np.asarray(static_scale, np.float32), (n,))
    p.scale.copy_(torch.tensor(np.array(init), dtype=torch.float32))
    p.quantize(dev(x16), dev(table), table.shape[1], static_scale=static_scale is not None)
    return p, p.scale


def _code_table(scale, fmt="e4m3"):
    """The oracle's byte for every fp16 bit pattern at this scale. The cast is
    elementwise, so table[bits(x)] is the oracle's quantize of x: full-size
    tensors are looked up instead of re-running the oracle on every element."""
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    with np.errstate(invalid="ignore"):          # the NaN and infinity patterns
        return fp8.quantize(allh, scale, fmt)


def _assert_every_record(pool, x16, table, scale, vl):
    """Every (block, kv head) record of a full-size pool against the oracle
    bytes, one batch row at a time (its blocks gathered on the device)."""
    import torch
    tab = _code_table(scale)
    b, h, s, d = x16.shape
    nbs = s // 16
    view = pool.view()
    for bi in range(b):
        nat = tab[x16[bi].view(np.uint16)].reshape(h, nbs, 16, d).transpose(1, 0, 2, 3)
        want = layout.fp8_pack_pool(nat, vl)
        got = host(view.index_select(0, torch.from_numpy(table[bi].astype(np.int64)).cuda()))
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)
            raise AssertionError(f"row {bi}: {len(bad)} bytes differ, first at {bad[:5].tolist()}")


def _oracle_decode_tab(q16, k16, v16, ks, vs, heads, q_fp8=False):
    """_oracle_decode for a per-tensor E4M3 scale with the keys and values
    quantized through the oracle's code tables (the same bytes, faster)."""
    b, hkv, s, d = k16.shape
    if q_fp8:
        q16 = fp8.query_hat(*fp8.quantize_query(q16))
    dec = fp8.decode(np.arange(256, dtype=np.uint8), "e4m3")
    ktab, vtab = _code_table(ks), _code_table(vs)
    kh = lambda bi, hi: dec[ktab[k16[bi, hi].view(np.uint16)]] * np.float64(ks)
    vh = lambda bi, hi: dec[vtab[v16[bi, hi].view(np.uint16)]] * np.float64(vs)
    return attention.decode_attention(q16, kh, vh, hkv, default_scale(d), heads)


def _wide_heads(w):
    """Two kv heads of every batch row, with all their query heads."""
    gq = w.q_heads // w.kv_heads
    out = []
    for bi in range(w.batch):
        for h in sorted({(3 * bi) % w.kv_heads, (3 * bi + 5) % w.kv_heads}):
            out += [(bi, h * gq + j) for j in range(gq)]
    return out


def _oracle_pool(x16, table, num_blocks, value_layout, scale, fmt="e4m3"):
    byts = fp8.quantize(x16, scale, fmt)
    nat = fp8.scatter_paged(byts, table, num_blocks, 16)
    return layout.fp8_pack_pool(nat, value_layout)


def test_all_fp16_values_cast_exactly():
    """Every fp16 bit pattern (finite and not) through the GPU cast at static scale 1."""
    allh = np.arange(65536, dtype=np.uint16).view(np.float16)
    x = allh.reshape(1, 4, 128, 128)                     # 4 kv heads x 128 tokens x 128 channels
    table = np.arange(8, dtype=np.int32).reshape(1, 8)
    for vl in (KEY, VALUE):
        pool, scale = _quantize(x, table, 8, vl, static_scale=1.0)
        want = _oracle_pool(x, table, 8, vl, np.float32(1.0))
        assert np.array_equal(host(pool.view()), want)


@pytest.mark.parametrize("special", [np.inf, -np.inf, np.nan])
def test_dynamic_scale_with_non_finite_values(special):
    """An infinity or NaN makes amax, hence the dynamic scale, non-finite; the
    cast then follows the formula with that scale (finite values go to zero,
    the special value to its saturated or NaN byte)."""
    x = workloads.make_inputs(1, 2, 4, 128, 32, 1, 5).k.copy()
    x[0, 1, 7, 33] = special
    table = np.arange(2, dtype=np.int32).reshape(1, 2)
    pool, scale = _quantize(x, table, 2, KEY)
    s_ref = fp8.dynamic_scale(x)
    got_s = host(scale)[0]
    assert (np.isnan(got_s) and np.isnan(s_ref)) or got_s == s_ref
    assert np.array_equal(host(pool.view()), _oracle_pool(x, table, 2, KEY, s_ref))


@pytest.mark.parametrize("d", [64, 128])
def test_dynamic_scale_and_bytes(d):
    rng = np.random.default_rng(d)
    x = workloads.make_inputs(3, 2, 4, d, 16 * 5 + 7, 1, 21).k          # ragged last block
    nb = 6
    table = rng.permutation(3 * nb + 4).astype(np.int32)[: 3 * nb].reshape(3, nb)
    pool, scale = _quantize(x, table, 3 * nb + 4, KEY)
    s_ref = fp8.dynamic_scale(x)
    assert host(scale)[0] == s_ref
    got = host(pool.view())
    want = _oracle_pool(x, table, 3 * nb + 4, KEY, s_ref)
    used = np.unique(table)
    assert np.array_equal(got[used], want[used])
    unused = np.setdiff1d(np.arange(3 * nb + 4), used)
    assert np.all(got[unused] == 0xAB)                   # untouched
    # the ragged last block's missing rows are zero bytes
    nat = layout.fp8_unpack_pool(got, d, KEY)
    assert np.all(nat[table[:, -1], :, 7:, :] == 0)


def test_saturation_with_static_scale():
    x = np.zeros((1, 1, 16, 64), np.float16)
    x[0, 0, 0, :4] = [1000, -700, 448, -465]
    x[0, 0, 1, :2] = [np.inf, -np.inf]
    table = np.zeros((1, 1), np.int32)
    pool, _ = _quantize(x, table, 1, KEY, static_scale=1.0)
    nat = layout.fp8_unpack_pool(host(pool.view()), 64, KEY)[0, 0]
    assert list(nat[0, :4]) == [0x7E, 0xFE, 0x7E, 0xFE]
    assert list(nat[1, :2]) == [0x7E, 0xFE]


def _decode(q16, kpool, vpool, kscale, vscale, table, seq_lens, hkv, num_blocks, max_seq, out_fp32=True,
            fmt="e4m3", per_head=False):
    import torch
    kvq = _kvq()
    b, hq, d = q16.shape
    out = torch.empty((b, hq, d), dtype=torch.float32 if out_fp32 else torch.float16, device="cuda")
    wsb = kvq.fp8_decode_workspace_bytes(b, hq, d)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    kvq.fp8_decode_attention(dev(q16), kpool.desc, vpool.desc, dev(table), dev(seq_lens.astype(np.int32)),
                             b, hq, table.shape[1], max_seq, out, out_fp32, 0.0, ws, wsb)
    return host(out).astype(np.float64), int(host(ws[:4].view(torch.int32))[0])


def _oracle_decode(q16, k16, v16, ks, vs, seq_lens, heads=None, fmt="e4m3", q_fp8=False):
    """ks, vs: scalars, or one scale per kv head; q_fp8: attention from the
    E4M3 query (FP8-domain attention)."""
    b, hkv, s, d = k16.shape
    if q_fp8:
        q16 = fp8.query_hat(*fp8.quantize_query(q16))
    ksh = lambda hi: np.float32(ks[hi] if np.ndim(ks) else ks)
    vsh = lambda hi: np.float32(vs[hi] if np.ndim(vs) else vs)
    kh = lambda bi, hi: fp8.decode(fp8.quantize(k16[bi, hi, : seq_lens[bi]], ksh(hi), fmt), fmt) * np.float64(ksh(hi))
    vh = lambda bi, hi: fp8.decode(fp8.quantize(v16[bi, hi, : seq_lens[bi]], vsh(hi), fmt), fmt) * np.float64(vsh(hi))
    return attention.decode_attention(q16, kh, vh, hkv, default_scale(d), heads)


@pytest.mark.parametrize("d,gq", [(128, 4), (64, 1), (128, 8), (64, 2), (128, 3), (64, 7)])
def test_decode_ragged_lengths(d, gq):
    rng = np.random.default_rng(d + gq)
    b, hkv, s = 3, 2, 16 * 40 + 9
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 31 + gq)
    nb = -(-s // 16)
    table = rng.permutation(b * nb).astype(np.int32).reshape(b, nb)
    kpool, kscale = _quantize(x.k, table, b * nb, KEY)
    vpool, vscale = _quantize(x.v, table, b * nb, VALUE)
    seq_lens = np.array([s, 1, 16 * 17 + 3])
    out, status = _decode(x.q[0], kpool, vpool, kscale, vscale, table, seq_lens, hkv, b * nb, s)
    ref = _oracle_decode(x.q[0], x.k, x.v, fp8.dynamic_scale(x.k), fp8.dynamic_scale(x.v), seq_lens)
    assert_attention_close(out, ref)
    assert status == 0
    out16, _ = _decode(x.q[0], kpool, vpool, kscale, vscale, table, seq_lens, hkv, b * nb, s, out_fp32=False)
    assert_attention_close(out16, ref, fp16_out=True)


def test_block_table_permutation_invariance():
    rng = np.random.default_rng(5)
    b, hkv, hq, d, s = 2, 2, 8, 128, 16 * 24
    x = workloads.make_inputs(b, hkv, hq, d, s, 1, 41)
    nb = s // 16
    ident = np.arange(b * nb, dtype=np.int32).reshape(b, nb)
    perm = rng.permutation(b * nb).astype(np.int32).reshape(b, nb)
    outs = []
    for table in (ident, perm):
        kpool, ks = _quantize(x.k, table, b * nb, KEY)
        vpool, vs = _quantize(x.v, table, b * nb, VALUE)
        outs.append(_decode(x.q[0], kpool, vpool, ks, vs, table, np.array([s, s]), hkv, b * nb, s)[0])
    assert np.array_equal(outs[0], outs[1])


def test_full_size_fp8_32k():
    """FP8 workload at full size: B 64, 8 kv heads, 32 q heads, D 128, 32768 tokens,
    blocks of 16 through a random permutation. Scales exact; every record of
    both pools exact; attention on 512 of the 2048 query heads."""
    import torch
    w = workloads.FP8_32K
    k, v, q, table = workloads.fp8_inputs(w)
    nb_total = w.batch * w.blocks_per_seq
    kpool, kscale = _quantize(k, table, nb_total, KEY)
    vpool, vscale = _quantize(v, table, nb_total, VALUE)
    ks_ref, vs_ref = fp8.dynamic_scale(k), fp8.dynamic_scale(v)
    assert host(kscale)[0] == ks_ref and host(vscale)[0] == vs_ref
    _assert_every_record(kpool, k, table, ks_ref, KEY)
    _assert_every_record(vpool, v, table, vs_ref, VALUE)
    seq_lens = np.full(w.batch, w.context)
    out, status = _decode(q, kpool, vpool, kscale, vscale, table, seq_lens, w.kv_heads, nb_total, w.context)
    assert status == 0
    heads = _wide_heads(w)
    ref = _oracle_decode_tab(q, k, v, ks_ref, vs_ref, heads)
    assert_attention_close(out, ref, heads)
    # the table route is the oracle's own arithmetic: one pair through the plain oracle agrees exactly
    one = heads[:4]
    assert np.array_equal(_oracle_decode(q, k, v, ks_ref, vs_ref, seq_lens, one)[tuple(np.array(one).T)],
                          ref[tuple(np.array(one).T)])
    del kpool, vpool
    torch.cuda.empty_cache()


# ------------------------------------------------------- E5M2 and per-head scales
def test_e5m2_all_fp16_values_cast_exactly():
    """Every fp16 bit pattern (finite and not) through the GPU E5M2 cast at static scale 1."""
    allh = np.arange(65536, dtype=np.uint16).view(np.float16)
    x = allh.reshape(1, 4, 128, 128)
    table = np.arange(8, dtype=np.int32).reshape(1, 8)
    for vl in (KEY, VALUE):
        pool, _ = _quantize(x, table, 8, vl, static_scale=1.0, fmt="e5m2")
        assert np.array_equal(host(pool.view()), _oracle_pool(x, table, 8, vl, np.float32(1.0), "e5m2"))


def _head_ranged_inputs(b, h, s, d, seed):
    x = workloads.make_inputs(b, h, 2 * h, d, s, 1, seed).k.astype(np.float32)
    ranges = np.array([0.002, 1.0, 40.0, 0.0, 900.0, 3.0, 0.3, 7.0][:h], np.float32)
    return (x * ranges.reshape(1, h, 1, 1)).astype(np.float16)     # one all-zero head


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("d", [64, 128])
def test_dynamic_per_head_scales_and_bytes(fmt, d):
    rng = np.random.default_rng(d + len(fmt))
    b, h, s = 3, 6, 16 * 5 + 7
    x = _head_ranged_inputs(b, h, s, d, 17)
    nb = 6
    table = rng.permutation(b * nb).astype(np.int32).reshape(b, nb)
    for vl in (KEY, VALUE):
        pool, scale = _quantize(x, table, b * nb, vl, fmt=fmt, per_head=True)
        s_ref = fp8.dynamic_scale_per_head(x, fmt)
        assert np.array_equal(host(scale), s_ref)
        assert np.array_equal(host(pool.view()), _oracle_pool(x, table, b * nb, vl, s_ref, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_static_per_head_scales(fmt):
    b, h, s, d = 2, 4, 48, 128
    x = _head_ranged_inputs(b, h, s, d, 23)
    table = np.arange(b * 3, dtype=np.int32).reshape(b, 3)
    given = np.array([1.0, 0.5, 0.01, 3.0e-5], np.float32)       # head 2 (|x| to ~150) saturates in E4M3
    pool, scale = _quantize(x, table, b * 3, KEY, static_scale=given, fmt=fmt, per_head=True)
    assert np.array_equal(host(scale), given)                     # read, not written
    assert np.array_equal(host(pool.view()), _oracle_pool(x, table, b * 3, KEY, given, fmt))


@pytest.mark.parametrize("special", [np.inf, np.nan])
def test_dynamic_e5m2_with_non_finite_values(special):
    x = workloads.make_inputs(1, 2, 4, 128, 32, 1, 6).k.copy()
    x[0, 0, 3, 9] = special
    table = np.arange(2, dtype=np.int32).reshape(1, 2)
    for per_head in (False, True):
        pool, scale = _quantize(x, table, 2, KEY, fmt="e5m2", per_head=per_head)
        s_ref = np.atleast_1d(fp8.dynamic_scale_per_head(x, "e5m2") if per_head else fp8.dynamic_scale(x, "e5m2"))
        got = host(scale)
        assert got.shape == s_ref.shape
        assert np.array_equal(np.isnan(got), np.isnan(s_ref)) and np.array_equal(got[~np.isnan(got)],
                                                                               s_ref[~np.isnan(got)])
        want = _oracle_pool(x, table, 2, KEY, s_ref if per_head else s_ref[0], "e5m2")
        assert np.array_equal(host(pool.view()), want)


@pytest.mark.parametrize("fmt,per_head", [("e5m2", False), ("e4m3", True), ("e5m2", True)])
@pytest.mark.parametrize("d,gq", [(128, 4), (64, 2), (128, 8)])
def test_decode_format_and_scale_variants(fmt, per_head, d, gq):
    rng = np.random.default_rng(d + gq + 31 * per_head)
    b, hkv, s = 3, 2, 16 * 30 + 9
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 61 + gq)
    k = (x.k.astype(np.float32) * np.array([1.0, 25.0]).reshape(1, 2, 1, 1)).astype(np.float16)
    nb = -(-s // 16)
    table = rng.permutation(b * nb).astype(np.int32).reshape(b, nb)
    kpool, kscale = _quantize(k, table, b * nb, KEY, fmt=fmt, per_head=per_head)
    vpool, vscale = _quantize(x.v, table, b * nb, VALUE, fmt=fmt, per_head=per_head)
    seq_lens = np.array([s, 1, 16 * 11 + 3])
    out, status = _decode(x.q[0], kpool, vpool, kscale, vscale, table, seq_lens, hkv, b * nb, s, fmt=fmt,
                          per_head=per_head)
    scale_of = fp8.dynamic_scale_per_head if per_head else fp8.dynamic_scale
    ref = _oracle_decode(x.q[0], k, x.v, scale_of(k, fmt), scale_of(x.v, fmt), seq_lens, fmt=fmt)
    assert_attention_close(out, ref)
    assert status == 0


# ------------------------------------------------------- FP8-domain attention (query in E4M3)
def _decode_qfp8(q16, kpool, vpool, kscale, vscale, table, seq_lens, hkv, num_blocks, max_seq, fmt="e4m3",
                 per_head=False, out_fp32=True):
    """fp8_decode_attention with q_fp8 = 1: (out, status word, E4M3 query bytes, query scale)
    read from the workspace at the offsets the header documents."""
    import torch
    kvq = _kvq()
    b, hq, d = q16.shape
    out = torch.empty((b, hq, d), dtype=torch.float32 if out_fp32 else torch.float16, device="cuda")
    wsb = kvq.fp8_decode_workspace_bytes(b, hq, d)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    kvq.fp8_decode_attention(dev(q16), kpool.desc, vpool.desc, dev(table), dev(seq_lens.astype(np.int32)),
                             b, hq, table.shape[1], max_seq, out, out_fp32, 0.0, ws, wsb, q_fp8=True)
    off = kvq.kv_decode_workspace_bytes(kvq.make_config(b, hq, hq, d, 2, 2, 128, 32))
    n = b * hq * d
    q8 = host(ws[off:off + n]).reshape(b, hq, d)
    qs_off = off + -(-n // 256) * 256
    q_scale = host(ws[qs_off:qs_off + 4].view(torch.float32))[0]
    return host(out).astype(np.float64), int(host(ws[:4].view(torch.int32))[0]), q8, q_scale


@pytest.mark.parametrize("d", [64, 128])
def test_key_pool_in_the_fp8_tensor_core_order(d):
    rng = np.random.default_rng(d + 5)
    x = workloads.make_inputs(2, 3, 6, d, 16 * 4 + 11, 1, 71).k
    nb = 5
    table = rng.permutation(2 * nb).astype(np.int32).reshape(2, nb)
    pool, scale = _quantize(x, table, 2 * nb, KEY)
    s_ref = fp8.dynamic_scale(x)
    assert host(scale)[0] == s_ref
    assert np.array_equal(host(pool.view()), _oracle_pool(x, table, 2 * nb, KEY, s_ref))


@pytest.mark.parametrize("fmt,per_head", [("e4m3", False), ("e5m2", False), ("e4m3", True), ("e5m2", True)])
@pytest.mark.parametrize("d,gq", [(128, 4), (64, 1), (128, 8), (64, 3)])
def test_fp8_domain_attention(fmt, per_head, d, gq):
    """q.k^T from the E4M3 query on FP8 tensor cores: the query bytes and scale
    are the oracle's bit for bit, attention is within the bars of the oracle
    on the same quantized query, keys and values."""
    rng = np.random.default_rng(d + gq + 7 * per_head)
    b, hkv, s = 3, 2, 16 * 30 + 9
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 81 + gq)
    k = (x.k.astype(np.float32) * np.array([1.0, 25.0]).reshape(1, 2, 1, 1)).astype(np.float16)
    q = (x.q[0].astype(np.float32) * 3.0).astype(np.float16)
    nb = -(-s // 16)
    table = rng.permutation(b * nb).astype(np.int32).reshape(b, nb)
    kpool, kscale = _quantize(k, table, b * nb, KEY, fmt=fmt, per_head=per_head)
    vpool, vscale = _quantize(x.v, table, b * nb, VALUE, fmt=fmt, per_head=per_head)
    seq_lens = np.array([s, 1, 16 * 11 + 3])
    out, status, q8, q_scale = _decode_qfp8(q, kpool, vpool, kscale, vscale, table, seq_lens, hkv, b * nb, s,
                                            fmt=fmt, per_head=per_head)
    codes_ref, scale_ref = fp8.quantize_query(q)
    assert q_scale == scale_ref
    assert np.array_equal(q8, codes_ref)
    scale_of = fp8.dynamic_scale_per_head if per_head else fp8.dynamic_scale
    ref = _oracle_decode(q, k, x.v, scale_of(k, fmt), scale_of(x.v, fmt), seq_lens, fmt=fmt, q_fp8=True)
    assert_attention_close(out, ref)
    assert status == 0


def test_fp8_domain_zero_query():
    """q = 0: scale 1, zero bytes, every score 0 — attention is the mean of the values."""
    b, hkv, gq, d, s = 2, 2, 4, 128, 16 * 7 + 5
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 91)
    nb = -(-s // 16)
    table = np.arange(b * nb, dtype=np.int32).reshape(b, nb)
    kpool, kscale = _quantize(x.k, table, b * nb, KEY)
    vpool, vscale = _quantize(x.v, table, b * nb, VALUE)
    q = np.zeros((b, hkv * gq, d), np.float16)
    seq_lens = np.array([s, 40])
    out, status, q8, q_scale = _decode_qfp8(q, kpool, vpool, kscale, vscale, table, seq_lens, hkv, b * nb, s)
    assert q_scale == 1.0 and not q8.any()
    vs = fp8.dynamic_scale(x.v)
    for bi in range(b):
        for h in range(hkv):
            vh = fp8.e4m3_decode(fp8.quantize(x.v[bi, h, :seq_lens[bi]], vs)).astype(np.float64) * float(vs)
            for hq in range(h * gq, (h + 1) * gq):
                assert np.allclose(out[bi, hq], vh.mean(axis=0), atol=2e-3, rtol=0)


def test_full_size_fp8_domain_attention_32k():
    """The 32K FP8 workload with the query in E4M3:
    scales and query bytes exact, attention on 512 of the 2048 query heads."""
    import torch
    w = workloads.FP8_32K
    k, v, q, table = workloads.fp8_inputs(w)
    nb_total = w.batch * w.blocks_per_seq
    kpool, kscale = _quantize(k, table, nb_total, KEY)
    vpool, vscale = _quantize(v, table, nb_total, VALUE)
    ks_ref, vs_ref = fp8.dynamic_scale(k), fp8.dynamic_scale(v)
    assert host(kscale)[0] == ks_ref and host(vscale)[0] == vs_ref
    rng = np.random.default_rng(4)
    for _ in range(12):
        b, h, j = int(rng.integers(w.batch)), int(rng.integers(w.kv_heads)), int(rng.integers(w.blocks_per_seq))
        want = layout.fp8_pack_pool(fp8.quantize(k[b, h, 16 * j:16 * j + 16], ks_ref)[None, None], KEY)[0, 0]
        assert np.array_equal(host(kpool.view()[table[b, j], h]), want)
    seq_lens = np.full(w.batch, w.context)
    out, status, q8, q_scale = _decode_qfp8(q, kpool, vpool, kscale, vscale, table, seq_lens, w.kv_heads,
                                            nb_total, w.context)
    assert status == 0
    codes_ref, scale_ref = fp8.quantize_query(q)
    assert q_scale == scale_ref and np.array_equal(q8, codes_ref)
    heads = _wide_heads(w)
    ref = _oracle_decode_tab(q, k, v, ks_ref, vs_ref, heads, q_fp8=True)
    assert_attention_close(out, ref, heads)
    del kpool, vpool
    torch.cuda.empty_cache()


def test_fp8_domain_fp16_output():
    rng = np.random.default_rng(93)
    b, hkv, gq, d, s = 2, 2, 4, 128, 16 * 20 + 3
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 94)
    nb = -(-s // 16)
    table = rng.permutation(b * nb).astype(np.int32).reshape(b, nb)
    kpool, kscale = _quantize(x.k, table, b * nb, KEY)
    vpool, vscale = _quantize(x.v, table, b * nb, VALUE)
    seq_lens = np.array([s, 100])
    out, status, q8, q_scale = _decode_qfp8(x.q[0], kpool, vpool, kscale, vscale, table, seq_lens, hkv, b * nb, s,
                                            out_fp32=False)
    ref = _oracle_decode(x.q[0], x.k, x.v, fp8.dynamic_scale(x.k), fp8.dynamic_scale(x.v), seq_lens, q_fp8=True)
    assert_attention_close(out, ref, fp16_out=True)
    assert status == 0


def test_decode_refuses_swapped_or_mismatched_pools():
    """The pools record their role, format and scale granularity; the decode
    refuses a value pool given as keys (and the reverse) and pools that disagree."""
    kvq = _kvq()
    b, hkv, gq, d, s = 1, 2, 2, 64, 32
    x = workloads.make_inputs(b, hkv, hkv * gq, d, s, 1, 97)
    table = np.arange(2, dtype=np.int32).reshape(1, 2)
    kpool, _ = _quantize(x.k, table, 2, KEY)
    vpool, _ = _quantize(x.v, table, 2, VALUE)
    v5, _ = _quantize(x.v, table, 2, VALUE, fmt="e5m2")
    vph, _ = _quantize(x.v, table, 2, VALUE, per_head=True)
    for kp, vp in ((vpool, kpool), (kpool, kpool), (kpool, v5), (kpool, vph)):
        with pytest.raises(kvq.KvqError) as e:
            _decode(x.q[0], kp, vp, None, None, table, np.array([s]), hkv, 2, s)
        assert e.value.name == "KVQ_ERR_ARG"
