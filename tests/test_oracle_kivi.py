"""Pins of the KIVI oracle: codes, scales, zero points and the streaming cache."""
import itertools

import numpy as np
import pytest

from oracle import kivi
from oracle.attention import decode_attention, default_scale


def _rand_groups(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


@pytest.mark.parametrize("bits", [2, 4])
def test_code_range(bits):
    rng = np.random.default_rng(0)
    x = _rand_groups(rng, (500, 32), 3.0)
    codes, s, z = kivi.quantize_groups(x, bits)
    assert codes.dtype == np.uint8
    assert codes.min() >= 0 and codes.max() <= 2 ** bits - 1
    # 2 bits have exactly four levels (CSDN page, section 11)
    assert set(np.unique(codes)) <= set(range(2 ** bits))


@pytest.mark.parametrize("bits", [2, 4])
def test_min_and_max_reconstruct(bits):
    rng = np.random.default_rng(1)
    x = _rand_groups(rng, (400, 32), 5.0)
    codes, s, z = kivi.quantize_groups(x, bits)
    xf = x.astype(np.float64)
    imin, imax = xf.argmin(-1), xf.argmax(-1)
    rows = np.arange(len(x))
    assert np.all(codes[rows, imin] == 0)
    assert np.all(codes[rows, imax] == 2 ** bits - 1)
    xh = kivi.dequantize(codes, s, z)
    assert np.array_equal(xh[rows, imin], xf[rows, imin])          # the min reconstructs exactly
    # the max is reconstructed up to the fp16 rounding of the scale
    err = np.abs(xh[rows, imax] - xf[rows, imax])
    assert np.all(err <= (2 ** bits - 1) * s.astype(np.float64) * 2.0 ** -11 + 1e-12)


@pytest.mark.parametrize("bits", [2, 4])
def test_round_trip_bound(bits):
    rng = np.random.default_rng(2)
    x = _rand_groups(rng, (2000, 32), 2.0)
    codes, s, z = kivi.quantize_groups(x, bits)
    xh = kivi.dequantize(codes, s, z)
    err = np.abs(xh - x.astype(np.float64))
    bound = s.astype(np.float64)[:, None] * (0.5 + 1e-6)
    assert np.all(err <= bound)


@pytest.mark.parametrize("bits", [2, 4])
def test_grid_inputs_round_trip_exactly(bits):
    """x_i = mn + k_i * s with s a power of two: codes equal k_i, dequantization is exact."""
    rng = np.random.default_rng(3)
    levels = 2 ** bits - 1
    for e in (-8, -3, 0, 2):
        s = 2.0 ** e
        k = rng.integers(0, levels + 1, size=(300, 32))
        k[:, 0], k[:, 1] = 0, levels                 # make the range exactly levels * s
        mn = np.float16(int(rng.integers(-64, 64)) * s)   # a multiple of s keeps every x exact
        x = (np.float64(mn) + k * s).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), np.float64(mn) + k * s)
        codes, s16, z16 = kivi.quantize_groups(x, bits)
        assert np.all(s16.astype(np.float64) == s)
        assert np.array_equal(codes, k)
        assert np.array_equal(kivi.dequantize(codes, s16, z16), x.astype(np.float64))


def test_brute_force_all_two_bit_vectors():
    """Every 2-bit code vector of four values on a grid: the quantizer recovers the
    closed form ``round((x - min) / ((max - min)/3))`` computed in exact rationals."""
    from fractions import Fraction
    s = 0.25
    for k in itertools.product(range(4), repeat=4):
        x = (np.float64(-1.0) + np.array(k) * s).astype(np.float16)
        codes, s16, z16 = kivi.quantize_groups(x[None], 2)
        lo, hi = min(k), max(k)
        if hi == lo:
            assert np.all(codes == 0)
            continue
        step = Fraction(hi - lo, 3) * Fraction(1, 4)       # exact (max - min) / 3
        step16 = Fraction(float(np.float16(float(step))))  # the stored fp16 scale
        assert Fraction(float(s16[0])) == step16
        for i, ki in enumerate(k):
            r = Fraction(ki - lo, 4) / step16
            fl = r.numerator // r.denominator
            rem = r - fl
            want = fl + (1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1) else 0)
            assert codes[0, i] == min(want, 3), (k, i)


def test_constant_group_and_underflowing_scale():
    x = np.full((1, 32), np.float16(1.5))
    codes, s, z = kivi.quantize_groups(x, 2)
    assert s[0] == 0 and np.all(codes == 0) and z[0] == np.float16(1.5)
    assert np.all(kivi.dequantize(codes, s, z) == 1.5)
    # range of one fp16 subnormal step: (2^-24)/3 rounds to 0 in fp16
    tiny = np.zeros((1, 32), np.float16)
    tiny[0, 5] = np.float16(2.0 ** -24)
    codes, s, z = kivi.quantize_groups(tiny, 2)
    assert s[0] == 0 and np.all(codes == 0)


def test_negative_zero_minimum_is_stored_as_plus_zero():
    x = np.zeros((1, 32), np.float16)
    x[0, 0] = np.float16(-0.0)
    x[0, 1] = np.float16(3.0)
    codes, s, z = kivi.quantize_groups(x, 2)
    assert z.view(np.uint16)[0] == 0


def test_key_axis_is_per_channel_and_value_axis_per_token():
    rng = np.random.default_rng(4)
    k = _rand_groups(rng, (2, 3, 64, 16))
    k[..., 5] *= 100                                   # an outlier channel
    codes, s, z = kivi.quantize_key_groups(k, 2)
    assert codes.shape == (2, 3, 2, 32, 16) and s.shape == (2, 3, 2, 16)
    # the channel-5 scale is set by channel 5 alone
    rng_ch = k[:, :, :32, 5].astype(np.float32)
    want = ((rng_ch.max(-1) - rng_ch.min(-1)) / np.float32(3)).astype(np.float16)
    assert np.array_equal(s[:, :, 0, 5], want)
    v = _rand_groups(rng, (2, 3, 64, 16))
    vc, vs, vz = kivi.quantize_value_tokens(v, 2)
    assert vc.shape == (2, 3, 2, 32, 16) and vs.shape == (2, 3, 2, 32)
    tok = v[1, 2, 40].astype(np.float32)
    assert vs[1, 2, 1, 8] == np.float16((tok.max() - tok.min()) / np.float32(3))


@pytest.mark.parametrize("s,r,want", [
    (256, 128, (128, 128)),        # tiny case: 4 groups + 128 residual
    (4096, 128, (3968, 128)),      # 4K case
    (8192, 128, (8064, 128)),      # 8K case
    (131072, 128, (130944, 128)),  # 128K streaming case
    (100, 128, (0, 100)),          # everything stays fp16
    (150, 128, (32, 118)),
    (4096, 0, (4096, 0)),          # R = 0: fully grouped storage
    (4100, 0, (4096, 4)),
])
def test_prefill_split(s, r, want):
    assert kivi.prefill_split(s, r) == want


def test_streaming_matches_prefill_for_shared_groups():
    rng = np.random.default_rng(5)
    b, h, d = 2, 2, 16
    k = _rand_groups(rng, (b, h, 256 + 200, d), 2.0)
    v = _rand_groups(rng, (b, h, 256 + 200, d), 2.0)
    c1 = kivi.KiviCache(b, h, d, 2, 2, 128)
    c1.prefill(k[:, :, :256], v[:, :, :256])
    for t in range(256, 456):
        c1.append(k[:, :, t], v[:, :, t])
    c2 = kivi.KiviCache(b, h, d, 2, 2, 128)
    c2.prefill(k, v)
    n = min(c1.k_codes.shape[2], c2.k_codes.shape[2])
    assert n >= 8
    for name in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero"):
        a, bb = getattr(c1, name)[:, :, :n], getattr(c2, name)[:, :, :n]
        assert np.array_equal(a.view(np.uint8), bb.view(np.uint8)), name
    # both hold the same tokens in the same order
    for bi in range(b):
        for hi in range(h):
            assert c1.keys_hat(bi, hi).shape[0] == 456 == c2.keys_hat(bi, hi).shape[0]


def test_flush_schedule_of_streaming_case():
    """128K case reduced in length: prefill leaves a full window, so the flush runs at
    steps 0, 128, 256, 384, each adding 4 groups."""
    rng = np.random.default_rng(6)
    c = kivi.KiviCache(1, 1, 16, 2, 2, 128)
    k = _rand_groups(rng, (1, 1, 256 + 512, 16))
    c.prefill(k[:, :, :256], k[:, :, :256])
    assert (c.n_grouped, c.n_resid) == (128, 128)
    flush_steps = []
    for step in range(512):
        before = c.n_grouped
        c.append(k[:, :, 256 + step], k[:, :, 256 + step])
        if c.n_grouped != before:
            assert c.n_grouped - before == 128
            flush_steps.append(step)
        assert 1 <= c.n_resid <= 128
    assert flush_steps == [0, 128, 256, 384]


def test_r0_streaming_flushes_every_group():
    rng = np.random.default_rng(7)
    c = kivi.KiviCache(1, 1, 16, 2, 2, residual=0)
    k = _rand_groups(rng, (1, 1, 100, 16))
    c.prefill(k[:, :, :64], k[:, :, :64])
    assert (c.n_grouped, c.n_resid) == (64, 0)
    for t in range(64, 100):
        c.append(k[:, :, t], k[:, :, t])
        assert c.n_resid == (t + 1) % 32
    assert c.n_grouped == 96


def test_capacity_is_enforced():
    c = kivi.KiviCache(1, 1, 16, 2, 2, 128, max_tokens=160)
    k = np.zeros((1, 1, 160, 16), np.float16)
    c.prefill(k, k)
    with pytest.raises(ValueError):
        c.append(k[:, :, 0], k[:, :, 0])


def test_short_context_equals_fp16_attention():
    """S <= R: nothing is quantized, so attention is plain fp16 attention
    (cross-checked with PyTorch's scaled_dot_product_attention in float64)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    b, hkv, hq, d, s = 2, 2, 8, 64, 100
    k = _rand_groups(rng, (b, hkv, s, d), 2.0)
    v = _rand_groups(rng, (b, hkv, s, d), 2.0)
    q = _rand_groups(rng, (b, hq, d))
    c = kivi.KiviCache(b, hkv, d, 2, 2, 128)
    c.prefill(k, v)
    assert c.n_grouped == 0
    scale = default_scale(d)
    out = decode_attention(q, c.keys_hat, c.values_hat, hkv, scale)
    kt = torch.from_numpy(k.astype(np.float64)).repeat_interleave(hq // hkv, dim=1)
    vt = torch.from_numpy(v.astype(np.float64)).repeat_interleave(hq // hkv, dim=1)
    qt = torch.from_numpy(q.astype(np.float64))[:, :, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=float(scale))[:, :, 0].numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_quantized_attention_error_follows_propagation_formula():
    """Score error equals q . eps / sqrt(d) (CSDN page, section 8.1) for the dequantized keys."""
    rng = np.random.default_rng(9)
    b, h, d = 1, 1, 64
    k = _rand_groups(rng, (b, h, 256, d), 2.0)
    c = kivi.KiviCache(b, h, d, 2, 2, 0)
    c.prefill(k, k)
    q = rng.standard_normal(d)
    kh = c.keys_hat(0, 0)
    eps = kh - k[0, 0].astype(np.float64)
    scale = 1 / np.sqrt(d)
    dscore = (kh @ q) * scale - (k[0, 0].astype(np.float64) @ q) * scale
    assert np.allclose(dscore, eps @ q * scale, atol=1e-9)
    # and is bounded by ||q||_1 * max|eps| / sqrt(d), max|eps| <= s/2
    smax = c.k_scale[0, 0].astype(np.float64).max()
    assert np.abs(dscore).max() <= np.abs(q).sum() * smax / 2 * scale * (1 + 1e-6)
