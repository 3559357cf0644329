"""Pins of the FP8 E4M3 oracle: the encoder, the per-tensor scale and the paged layout."""
import numpy as np
import pytest

from oracle import fp8


def _finite_e4m3_table():
    """The 254 finite E4M3 values from the bit layout, by exhaustive listing."""
    vals = {}
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e, m = (b >> 3) & 15, b & 7
        if e == 15 and m == 7:
            continue
        vals[b] = s * (m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return vals


def _brute_force_encode(y):
    """Nearest finite E4M3 value, ties to the even code, saturating at +-448, NaN -> 0x7F."""
    table = _finite_e4m3_table()
    pos = sorted((v, b) for b, v in table.items() if v >= 0 and not (b & 0x80))
    vals = np.array([v for v, _ in pos])
    codes = np.array([b for _, b in pos])
    y = np.asarray(y, np.float64)
    out = np.empty(y.shape, np.uint8)
    for i, v in enumerate(y.ravel()):
        if np.isnan(v):
            out.flat[i] = 0x7F
            continue
        sgn = 0x80 if np.signbit(v) else 0
        a = min(abs(v), 448.0)
        dist = np.abs(vals - a)
        best = np.flatnonzero(dist == dist.min())
        if len(best) > 1:
            best = [j for j in best if codes[j] % 2 == 0]
        out.flat[i] = codes[best[0]] | sgn
    return out


def test_format_facts():
    table = _finite_e4m3_table()
    assert len(table) == 254
    assert max(table.values()) == 448.0               # the E4M3 max used for the scale
    assert min(v for v in table.values() if v > 0) == 2.0 ** -9
    dec = fp8.e4m3_decode(np.arange(256))
    for b in range(256):
        if b in table:
            assert dec[b] == table[b]
        else:
            assert np.isnan(dec[b])


def test_all_fp16_inputs_against_brute_force():
    x = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    got = fp8.e4m3_encode(x)
    want = _brute_force_encode(x)
    assert np.array_equal(got, want)


def test_against_torch_float8_cast():
    torch = pytest.importorskip("torch")
    x = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 448)]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), ref)


def test_saturation_nan_and_signed_zero():
    y = np.array([448, 464, 465, 1e10, np.inf, -np.inf, -470, np.nan, -np.nan, -0.0, 0.0], np.float32)
    got = fp8.e4m3_encode(y)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x7F, 0x80, 0x00]


def test_ties_and_subnormals():
    y = np.array([2.0 ** -10, 1.5 * 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -6 * (1 + 1 / 16), 2.0 ** -6 * 1.1875], np.float32)
    got = fp8.e4m3_encode(y)
    # 2^-10 is the tie between 0 and 2^-9 -> 0 (even); 1.5*2^-10 -> 2^-9 (code 1);
    # 3*2^-10 is the tie between 2^-9 and 2*2^-9 -> code 2 (even);
    # 2^-6*(1+1/16) is the tie between codes 8 and 9 -> 8; 2^-6*1.1875 is the tie between
    # codes 9 and 10 -> 10
    assert list(got) == [0, 1, 2, 8, 10]


def test_dynamic_scale_amax_over_448():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((4, 3, 50, 16)) * 7).astype(np.float16)
    s = fp8.dynamic_scale(x)
    a = np.abs(x.astype(np.float32)).max()
    assert s == np.float32(a / np.float32(448.0))
    q = fp8.quantize(x, s)
    idx = np.unravel_index(np.abs(x.astype(np.float32)).argmax(), x.shape)
    # the amax element always lands on the largest code
    assert q[idx] in (0x7E, 0xFE)
    # every code is finite and within +-448
    dec = fp8.e4m3_decode(q)
    assert np.all(np.isfinite(dec)) and np.all(np.abs(dec) <= 448)
    # a tensor whose amax is 448 gets scale 1 (the worked code on the yunthe page)
    y = np.array([448, -3, 1], np.float16)
    assert fp8.dynamic_scale(y) == 1.0
    assert fp8.dynamic_scale(np.zeros(8, np.float16)) == 1.0


def test_relative_error_bound():
    """Normal-range E4M3 rounding error is at most 2^-4 relative."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * 3).astype(np.float16)
    s = fp8.dynamic_scale(x)
    xh = fp8.e4m3_decode(fp8.quantize(x, s)) * np.float64(s)
    xf = x.astype(np.float64)
    normal = np.abs(xf / s) >= 2.0 ** -6
    assert np.all(np.abs(xh - xf)[normal] <= np.abs(xf)[normal] * 2.0 ** -4 * (1 + 1e-12))


def test_static_scale_one_saturates():
    x = np.array([1000, -700, 3.3, 0.001], np.float16)
    q = fp8.quantize(x, np.float32(1.0))
    assert q[0] == 0x7E and q[1] == 0xFE


def test_paged_scatter_gather():
    rng = np.random.default_rng(2)
    b, h, s, d, bs = 3, 2, 50, 8, 16
    byts = rng.integers(0, 256, size=(b, h, s, d), dtype=np.uint8)
    nb = -(-s // bs)
    table = rng.permutation(b * nb).astype(np.int32).reshape(b, nb)
    pool = fp8.scatter_paged(byts, table, b * nb, bs)
    for bi in range(b):
        for hi in range(h):
            assert np.array_equal(fp8.gather_paged(pool, table, bi, hi, s), byts[bi, hi])
    ident = np.arange(b * nb, dtype=np.int32).reshape(b, nb)
    pool2 = fp8.scatter_paged(byts, ident, b * nb, bs)
    # identity table: block bi*nb + j holds tokens 16j.. of sequence bi
    assert np.array_equal(pool2[1 * nb + 2, 1, :, :], byts[1, 1, 32:48])
    # one byte per element: half of fp16
    assert pool[:, :, :, :].size == b * nb * h * bs * d


# ---------------------------------------------------------------- E5M2
def _finite_e5m2_table():
    """The finite E5M2 values from the bit layout, by exhaustive listing."""
    vals = {}
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e, m = (b >> 2) & 31, b & 3
        if e == 31:
            continue
        vals[b] = s * (m / 4 * 2.0 ** -14 if e == 0 else (1 + m / 4) * 2.0 ** (e - 15))
    return vals


def test_e5m2_format_facts():
    table = _finite_e5m2_table()
    assert len(table) == 248
    assert max(table.values()) == fp8.E5M2_MAX == 57344.0
    assert min(v for v in table.values() if v > 0) == 2.0 ** -16
    dec = fp8.e5m2_decode(np.arange(256))
    for b in range(256):
        if b in table:
            assert dec[b] == table[b]
    assert np.isinf(dec[0x7C]) and np.isinf(dec[0xFC]) and np.isnan(dec[0x7D]) and np.isnan(dec[0xFF])


def test_e5m2_all_fp16_inputs_against_brute_force():
    table = _finite_e5m2_table()
    pos = sorted((v, b) for b, v in table.items() if v >= 0 and not (b & 0x80))
    vals = np.array([v for v, _ in pos])
    codes = np.array([b for _, b in pos])
    x = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    got = fp8.e5m2_encode(x)
    for i, v in enumerate(x.astype(np.float64)):
        if np.isnan(v):
            assert got[i] == 0x7F
            continue
        sgn = 0x80 if np.signbit(v) else 0
        a = min(abs(v), fp8.E5M2_MAX)
        dist = np.abs(vals - a)
        best = np.flatnonzero(dist == dist.min())
        if len(best) > 1:
            best = [j for j in best if codes[j] % 2 == 0]
        assert got[i] == codes[best[0]] | sgn, (i, v)


def test_e5m2_is_fp16_rounded_to_its_top_byte():
    """E5M2 shares fp16's sign and exponent fields: below the saturation point
    the code is the fp16 bit pattern rounded to its top byte, ties to even."""
    bits = np.arange(65536, dtype=np.uint32)
    x = bits.astype(np.uint16).view(np.float16)
    ok = np.isfinite(x) & (np.abs(x.astype(np.float64)) < 57344.0)
    mag = bits & 0x7FFF
    rounded = (mag + 0x7F + ((mag >> 8) & 1)) >> 8            # round the low 8 bits, ties to even
    want = (rounded | ((bits >> 8) & 0x80)).astype(np.uint8)
    got = fp8.e5m2_encode(x.astype(np.float32))
    assert np.array_equal(got[ok], want[ok])


def test_e5m2_against_torch_cast():
    torch = pytest.importorskip("torch")
    x = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 57344)]
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e5m2_encode(x), ref)


def test_e5m2_saturation_nan_and_signed_zero():
    y = np.array([57344, 61439, 61440, 1e10, np.inf, -np.inf, -70000, np.nan, -0.0, 0.0], np.float32)
    assert list(fp8.e5m2_encode(y)) == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0xFB, 0x7F, 0x80, 0x00]


def test_e5m2_dynamic_scale():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2, 3, 40, 16)) * 900).astype(np.float16)
    s = fp8.dynamic_scale(x, "e5m2")
    assert s == np.float32(np.float32(np.abs(x.astype(np.float32)).max()) / np.float32(57344.0))
    q = fp8.quantize(x, s, "e5m2")
    idx = np.unravel_index(np.abs(x.astype(np.float32)).argmax(), x.shape)
    assert q[idx] in (0x7B, 0xFB)
    dec = fp8.e5m2_decode(q)
    assert np.all(np.isfinite(dec)) and np.all(np.abs(dec) <= 57344)


# ---------------------------------------------------------------- per-head scales
def test_per_head_scales_follow_each_head():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 4, 33, 16)).astype(np.float32)
    x *= np.array([0.01, 1.0, 30.0, 0.0]).reshape(1, 4, 1, 1)       # very different ranges, one all-zero head
    x = x.astype(np.float16)
    for fmt in fp8.FORMATS:
        sh = fp8.dynamic_scale_per_head(x, fmt)
        assert sh.shape == (4,) and sh.dtype == np.float32
        for h in range(4):
            a = np.float32(np.abs(x[:, h].astype(np.float32)).max())
            assert sh[h] == (np.float32(1.0) if a == 0 else np.float32(a / np.float32(fp8.fmax(fmt))))
        q = fp8.quantize(x, sh, fmt)
        for h in range(4):                                            # per-head == per-slice scalar
            assert np.array_equal(q[:, h], fp8.quantize(x[:, h], sh[h], fmt))
        # each nonzero head reaches the format's largest code, which one per-tensor scale would not
        for h in range(3):
            assert np.max(q[:, h] & 0x7F) == (0x7E if fmt == "e4m3" else 0x7B)


def test_query_on_the_grid_is_unchanged():
    """A query whose values are E4M3 values with amax exactly 448 has scale 1,
    and FP8-domain attention then uses the query itself."""
    rng = np.random.default_rng(11)
    grid = fp8.e4m3_decode(np.arange(0x7F, dtype=np.uint8))      # every finite non-negative E4M3 value
    q = rng.choice(grid, size=(2, 4, 64)) * rng.choice([-1.0, 1.0], size=(2, 4, 64))
    q[0, 0, 0] = 448.0
    q16 = q.astype(np.float16)
    codes, scale = fp8.quantize_query(q16)
    assert scale == np.float32(1.0)
    assert np.array_equal(fp8.query_hat(codes, scale), q16.astype(np.float64))


def test_query_quantization_error_bound():
    """Every quantized query element is within half an E4M3 step of q/scale:
    2^-4 relative in the normal range, 2^-10 absolute below it (half the
    smallest subnormal, 2^-9); the largest magnitude lands on +-448."""
    rng = np.random.default_rng(12)
    q16 = (rng.standard_normal((4, 8, 128)) * rng.lognormal(0, 1, size=(4, 8, 1))).astype(np.float16)
    codes, scale = fp8.quantize_query(q16)
    y = q16.astype(np.float64) / float(scale)
    yh = fp8.e4m3_decode(codes).astype(np.float64)
    bound = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(np.abs(yh - y) <= bound)
    i = np.unravel_index(np.argmax(np.abs(q16.astype(np.float64))), q16.shape)
    assert codes[i] in (0x7E, 0xFE)
    z_codes, z_scale = fp8.quantize_query(np.zeros((1, 2, 64), np.float16))
    assert z_scale == np.float32(1.0) and not z_codes.any()
