"""GPU parity of the NVFP4 paged path against the CPU oracle, through the C ABI.

Pool bytes (codes and block scales, in the in-block order of each role) and
the tensor scale must match bit for bit; attention must stay within max-abs
2e-3 and relative L2 1e-3 of the float64 oracle computed on the same
dequantized values.
"""
import numpy as np
import pytest

from oracle import attention, fp8, layout, nvfp4
from oracle.attention import default_scale
from quantized_kv_cache_quant_gb300 import workloads

from kvq_helpers import assert_attention_close, dev, host

pytestmark = pytest.mark.gpu


def _kvq():
    from quantized_kv_cache_quant_gb300 import kvq
    return kvq


def _pool(role, x16, table, num_blocks, static_scale=None):
    import torch
    kvq = _kvq()
    b, h, s, d = x16.shape
    p = kvq.Nvfp4Pool(role, num_blocks, h, d)
    p.buf.fill_(0xAB)
    if static_scale is not None:
        p.scale[0] = float(static_scale)
    else:
        p.scale[0] = -1.0
    p.quantize(dev(x16), dev(table), table.shape[1], static_scale=static_scale is not None)
    torch.cuda.synchronize()
    return p


def _oracle_pool(role, x16, table, num_blocks, s_t):
    codes, sb = nvfp4.quantize(x16, s_t)
    cp = fp8.scatter_paged(codes, table, num_blocks, 16)
    sp = fp8.scatter_paged(sb, table, num_blocks, 16)
    return layout.nvfp4_pack_pool(cp, sp, role)


def _assert_pool(p, want, touched):
    got = host(p.view())
    assert np.array_equal(got[touched], want[touched]), \
        f"{np.count_nonzero(got[touched] != want[touched])} bytes differ"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("role", [0, 1])
def test_quantize_bytes_dynamic_scale(d, role):
    kvq = _kvq()
    b, h, s = 2, 3, 100                        # 7 blocks per sequence, the last one ragged
    x = workloads.make_inputs(b, h, h, d, s, 1, 31 + d + role)
    x16 = x.k if role == kvq.ROLE_KEY else x.v
    nb = -(-s // 16)
    table = workloads.block_table(b, nb, 32)
    p = _pool(role, x16, table, b * nb)
    s_t = nvfp4.tensor_scale(x16)
    assert host(p.scale)[0] == s_t
    _assert_pool(p, _oracle_pool(role, x16, table, b * nb, s_t), table.ravel())


@pytest.mark.parametrize("role", [0, 1])
def test_every_fp16_value_through_the_cast(role):
    """Every finite fp16 value at a static tensor scale of 1: E2M1 rounding and the
    E4M3 block scale over the whole fp16 range (blocks mix neighbouring values)."""
    allh = np.arange(65536, dtype=np.uint16).view(np.float16)
    allh = np.where(np.isfinite(allh), allh, np.float16(0))
    x = allh.reshape(1, 4, 128, 128)
    table = np.arange(8, dtype=np.int32).reshape(1, 8)
    p = _pool(role, x, table, 8, static_scale=1.0)
    _assert_pool(p, _oracle_pool(role, x, table, 8, np.float32(1.0)), np.arange(8))


def test_static_scale_saturation():
    """A static scale far below the data's: block scales saturate at 448 and codes at +-6."""
    kvq = _kvq()
    x = workloads.make_inputs(1, 2, 2, 128, 48, 1, 40).k
    table = np.arange(3, dtype=np.int32).reshape(1, 3)
    s_t = np.float32(1e-3)
    p = _pool(kvq.ROLE_KEY, x, table, 3, static_scale=s_t)
    assert host(p.scale)[0] == s_t
    _assert_pool(p, _oracle_pool(kvq.ROLE_KEY, x, table, 3, s_t), np.arange(3))


@pytest.mark.parametrize("s_t", [2.0 ** -110, 1.0 / 64])
@pytest.mark.parametrize("role", [0, 1])
def test_zero_blocks_negative_zeros_and_the_division_path(role, s_t):
    """A static tensor scale of 2^-110 puts every nonzero block divisor
    fl32(S_b * s_t) below 2^-96, where the cast takes the IEEE division (the
    whole unit); 1/64 keeps the reciprocal path. All-zero and negative-zero
    blocks give codes 0 either way, and a negative zero in a nonzero block keeps
    its sign (code 8)."""
    x = workloads.make_inputs(1, 2, 2, 128, 48, 1, 41).v.astype(np.float16)
    x[0, 0, 5] = 0.0                             # a zero token: every block of it 0
    x[0, 1, 7] = np.float16(-0.0)                # a negative-zero token
    x[0, 1, 20, :16] = np.float16(-0.0)          # one negative-zero block in a token
    x[0, 1, 21, 3] = np.float16(-0.0)            # a negative zero in a nonzero block: code 8
    table = np.arange(3, dtype=np.int32).reshape(1, 3)
    s_t = np.float32(s_t)
    p = _pool(role, x, table, 3, static_scale=s_t)
    want = _oracle_pool(role, x, table, 3, s_t)
    _assert_pool(p, want, np.arange(3))
    codes, sb = nvfp4.quantize(x, s_t)
    divisors = fp8.e4m3_decode(sb[sb != 0]) * float(s_t)
    assert np.any(codes == 8)
    assert np.all(divisors < 2.0 ** -96) if s_t < 2.0 ** -100 else np.all(divisors >= 2.0 ** -96)


def test_table_entries_outside_the_pool_are_skipped():
    kvq = _kvq()
    x = workloads.make_inputs(1, 2, 2, 64, 48, 1, 41).v
    table = np.array([[0, 5, 2]], np.int32)   # 5 is outside a 3-block pool
    p = _pool(kvq.ROLE_VALUE, x, table, 3)
    got = host(p.view())
    assert np.all(got[1] == 0xAB)              # untouched
    want = _oracle_pool(kvq.ROLE_VALUE, x[:, :, :16], np.array([[0]], np.int32), 3, nvfp4.tensor_scale(x))
    assert np.array_equal(got[0], want[0])


def _decode(x, table, nb, lens, q_heads, out_fp32=True, scale=0.0):
    import torch
    kvq = _kvq()
    b, h, s, d = x.k.shape
    k = _pool(kvq.ROLE_KEY, x.k, table, b * nb)
    v = _pool(kvq.ROLE_VALUE, x.v, table, b * nb)
    out = torch.empty((b, q_heads, d), dtype=torch.float32 if out_fp32 else torch.float16, device="cuda")
    wsb = kvq.nvfp4_decode_workspace_bytes(b, q_heads, d)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    kvq.nvfp4_decode_attention(dev(x.q[0]), k.desc, v.desc, dev(table), dev(lens), b, q_heads, nb, int(lens.max()),
                               out, out_fp32, scale, ws, wsb)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    return host(out).astype(np.float64)


def _oracle_decode(x, lens, heads=None, scale=None):
    b, h, s, d = x.k.shape
    kt, vt = nvfp4.tensor_scale(x.k), nvfp4.tensor_scale(x.v)
    kc, ksb = nvfp4.quantize(x.k, kt)
    vc, vsb = nvfp4.quantize(x.v, vt)
    kh = lambda bi, hi: nvfp4.dequantize(kc[bi, hi, :lens[bi]], ksb[bi, hi, :lens[bi]], kt)
    vh = lambda bi, hi: nvfp4.dequantize(vc[bi, hi, :lens[bi]], vsb[bi, hi, :lens[bi]], vt)
    return attention.decode_attention(x.q[0], kh, vh, h, default_scale(d) if scale is None else scale, heads)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("gq", [1, 2, 3, 4, 8])
def test_decode_attention(d, gq):
    b, h, s = 3, 2, 300
    x = workloads.make_inputs(b, h, h * gq, d, s, 1, 50 + d + gq)
    nb = -(-s // 16)
    table = workloads.block_table(b, nb, 51)
    lens = np.array([300, 17, 161], np.int32)
    got = _decode(x, table, nb, lens, h * gq)
    assert_attention_close(got, _oracle_decode(x, lens))


@pytest.mark.parametrize("gq", [4, 8])
def test_decode_rising_logits(gq):
    """Keys that drift along the query heads' mean direction, so each head's
    logits rise through the sequence (by 6 to 25 in log2 units over a spread
    of about 4.5 between tokens): the running maximum of the decode moves many
    times, in steps below and above its slack, in both operand arrangements (at most 4 query heads per kv
    head: tokens on the tile rows; more: heads on the rows)."""
    b, h, s, d = 2, 2, 16 * 37 + 9, 128
    x = workloads.make_inputs(b, h, h * gq, d, s, 1, 70 + gq)
    k = x.k.astype(np.float64)
    q = x.q[0].astype(np.float64)
    for bi in range(b):
        for hi in range(h):
            u = q[bi, hi * gq:(hi + 1) * gq].sum(axis=0)
            u /= np.linalg.norm(u)
            k[bi, hi] += np.linspace(0.0, 24.0, s)[:, None] * u
    xs = workloads.KVInputs(k.astype(np.float16), x.v, x.q, x.k_new, x.v_new)
    nb = -(-s // 16)
    table = workloads.block_table(b, nb, 71)
    lens = np.array([s, 16 * 20 + 3], np.int32)
    got = _decode(xs, table, nb, lens, h * gq)
    assert_attention_close(got, _oracle_decode(xs, lens))


def test_decode_fp16_output_and_custom_scale():
    b, h, s, d = 2, 2, 64, 128
    x = workloads.make_inputs(b, h, 8, d, s, 1, 60)
    table = workloads.block_table(b, 4, 61)
    lens = np.array([64, 33], np.int32)
    got = _decode(x, table, 4, lens, 8, out_fp32=False, scale=0.05)
    assert_attention_close(got, _oracle_decode(x, lens, scale=np.float32(0.05)), fp16_out=True)


@pytest.mark.slow
def test_full_size_nvfp4_32k():
    """The 32K workload: the tensor scales, every byte of sampled blocks of both
    pools, and attention on sampled query heads against the oracle."""
    import torch
    kvq = _kvq()
    w = workloads.NVFP4_32K
    k16, v16, q, table = workloads.fp8_inputs(w)
    nb = w.blocks_per_seq
    k = _pool(kvq.ROLE_KEY, k16, table, w.batch * nb)
    v = _pool(kvq.ROLE_VALUE, v16, table, w.batch * nb)
    kt, vt = nvfp4.tensor_scale(k16), nvfp4.tensor_scale(v16)
    assert host(k.scale)[0] == kt and host(v.scale)[0] == vt
    rng = np.random.default_rng(0)
    for bi in rng.choice(w.batch, 4, replace=False):
        for pool, x16, s_t, role in ((k, k16, kt, 0), (v, v16, vt, 1)):
            for j in rng.choice(nb, 6, replace=False):
                codes, sb = nvfp4.quantize(x16[bi, :, 16 * j:16 * j + 16], s_t)   # [H, 16, D], [H, 16, D/16]
                got = host(pool.view()[int(table[bi, j])])
                for hh in range(w.kv_heads):
                    assert np.array_equal(got[hh], layout.nvfp4_pack_record(codes[hh], sb[hh], role)), (bi, j, hh)
    out = torch.empty((w.batch, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    wsb = kvq.nvfp4_decode_workspace_bytes(w.batch, w.q_heads, w.head_dim)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    lens = np.full(w.batch, w.context, np.int32)
    kvq.nvfp4_decode_attention(dev(q), k.desc, v.desc, dev(table), dev(lens), w.batch, w.q_heads, nb, w.context,
                               out, True, 0.0, ws, wsb)
    torch.cuda.synchronize()
    heads = [(int(bi), int(hq)) for bi, hq in zip(rng.choice(w.batch, 6), rng.choice(w.q_heads, 6))]

    def deq(x16, s_t):
        return lambda bi, hi: nvfp4.dequantize(*nvfp4.quantize(x16[bi, hi], s_t), s_t)

    ref = attention.decode_attention(q, deq(k16, kt), deq(v16, vt), w.kv_heads, default_scale(w.head_dim), heads)
    assert_attention_close(host(out), ref, heads=heads)
