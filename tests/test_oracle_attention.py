"""Pins of the float64 decode-attention oracle."""
import numpy as np
import pytest

from oracle import attention, fp8, kivi


def test_against_torch_sdpa_gqa():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    b, hkv, hq, t, d = 2, 2, 8, 37, 16
    k = rng.standard_normal((b, hkv, t, d))
    v = rng.standard_normal((b, hkv, t, d))
    q = rng.standard_normal((b, hq, d))
    out = attention.decode_attention(q, lambda bi, hi: k[bi, hi], lambda bi, hi: v[bi, hi], hkv, 0.3)
    kt = torch.from_numpy(k).repeat_interleave(hq // hkv, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(hq // hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[:, :, None], kt, vt, scale=0.3)
    assert np.allclose(out, ref[:, :, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    k, v, q = rng.standard_normal((1, 8)), rng.standard_normal((1, 8)), rng.standard_normal(8)
    assert np.array_equal(attention.softmax_attend(q, k, v, 0.5), v[0])


def test_zero_query_or_identical_keys_give_the_mean():
    rng = np.random.default_rng(2)
    k, v = rng.standard_normal((9, 8)), rng.standard_normal((9, 8))
    assert np.allclose(attention.softmax_attend(np.zeros(8), k, v, 1.0), v.mean(0), rtol=1e-13, atol=1e-13)
    kk = np.repeat(k[:1], 9, axis=0)
    assert np.allclose(attention.softmax_attend(rng.standard_normal(8), kk, v, 1.0), v.mean(0), rtol=1e-13, atol=1e-13)


def test_gqa_sharing_and_mha_reduction():
    rng = np.random.default_rng(3)
    b, hkv, t, d = 1, 2, 20, 8
    k, v = rng.standard_normal((b, hkv, t, d)), rng.standard_normal((b, hkv, t, d))
    q1 = rng.standard_normal((b, 1, d))
    q = np.repeat(q1, 8, axis=1)                         # identical queries in both groups
    out = attention.decode_attention(q, lambda bi, hi: k[bi, hi], lambda bi, hi: v[bi, hi], hkv, 0.4)
    assert np.all(out[0, :4] == out[0, :1]) and np.all(out[0, 4:] == out[0, 4:5])
    assert [attention.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    mha = attention.decode_attention(q[:, :2], lambda bi, hi: k[bi, hi], lambda bi, hi: v[bi, hi], hkv, 0.4)
    assert np.array_equal(mha[0, 0], out[0, 0]) and np.array_equal(mha[0, 1], out[0, 4])


def test_token_order_and_block_permutation_invariance():
    rng = np.random.default_rng(4)
    t, d = 64, 8
    k, v, q = rng.standard_normal((t, d)), rng.standard_normal((t, d)), rng.standard_normal(d)
    perm = rng.permutation(t)
    a = attention.softmax_attend(q, k, v, 0.7)
    bb = attention.softmax_attend(q, k[perm], v[perm], 0.7)
    assert np.allclose(a, bb, rtol=1e-13, atol=1e-13)
    # paged FP8 cache: the same bytes through two different block tables give the same tokens
    byts = rng.integers(0, 126, size=(1, 1, 48, d), dtype=np.uint8)
    t1 = np.array([[2, 0, 1]], np.int32)
    t2 = np.array([[0, 1, 2]], np.int32)
    g1 = fp8.gather_paged(fp8.scatter_paged(byts, t1, 3, 16), t1, 0, 0, 48)
    g2 = fp8.gather_paged(fp8.scatter_paged(byts, t2, 3, 16), t2, 0, 0, 48)
    assert np.array_equal(g1, g2)


def test_brute_force_tiny_quantized_cache():
    """Tiny KIVI cache: attention over the dequantized tokens equals an explicit
    double loop over tokens with math.exp."""
    import math
    rng = np.random.default_rng(5)
    k = (rng.standard_normal((1, 1, 40, 16)) * 3).astype(np.float16)
    v = rng.standard_normal((1, 1, 40, 16)).astype(np.float16)
    c = kivi.KiviCache(1, 1, 16, 2, 2, 0)
    c.prefill(k, v)
    assert (c.n_grouped, c.n_resid) == (32, 8)
    q = rng.standard_normal(16)
    kh, vh = c.keys_hat(0, 0), c.values_hat(0, 0)
    got = attention.softmax_attend(q, kh, vh, 0.25)
    scores = [sum(q[j] * kh[i, j] for j in range(16)) * 0.25 for i in range(40)]
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    z = sum(w)
    want = [sum(w[i] * vh[i, j] for i in range(40)) / z for j in range(16)]
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    # grouped tokens dequantize to code * scale + zero, residual tokens are the fp16 inputs
    assert np.array_equal(kh[32:], k[0, 0, 32:].astype(np.float64))
    assert np.array_equal(kh[:32, 3], c.k_codes[0, 0, 0, :, 3] * np.float64(c.k_scale[0, 0, 0, 3]) + np.float64(c.k_zero[0, 0, 0, 3]))
