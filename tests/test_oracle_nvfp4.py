"""Pins of the NVFP4 oracle (E2M1 values, E4M3 block scales, fp32 tensor scale).

Each pin checks the oracle against something other than itself: a brute-force
nearest-value search over every fp16 input, the bit-field table of the
format, hand-made blocks whose exact result is known, and error bounds that
follow from the grid.
"""
import numpy as np
import pytest

from oracle import fp8, nvfp4

MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_bit_fields():
    codes = np.arange(16, dtype=np.uint8)
    want = np.array(MAGS + [-m for m in MAGS])
    got = nvfp4.e2m1_decode(codes)
    assert np.array_equal(got, want)
    assert np.signbit(got[8])  # code 8 is -0


def _brute_force(y: float) -> int:
    """Nearest E2M1 value with ties to the even code, same sign, saturating."""
    neg = np.signbit(np.float32(y))
    a = abs(float(y))
    if a > 6.0:
        return 7 | (8 if neg else 0)
    dist = [abs(a - m) for m in MAGS]
    best = min(dist)
    cands = [c for c in range(8) if dist[c] == best]
    if len(cands) > 1:
        cands = [c for c in cands if c % 2 == 0]
    assert len(cands) == 1
    return cands[0] | (8 if neg else 0)


def test_e2m1_encode_every_fp16_value():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16)
    finite = np.isfinite(x)
    y = x[finite].astype(np.float32)
    got = nvfp4.e2m1_encode(y)
    # the brute force only needs the distinct magnitudes around the grid; evaluate it per value
    want = np.array([_brute_force(v) for v in y.tolist()], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(y[i]), int(got[i]), int(want[i])) for i in bad[:10]]


def test_e2m1_ties_and_saturation():
    y = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.5, 6.0, 6.5, 1e30, -0.25, -5.0, -7.0], np.float32)
    want = np.array([0, 2, 2, 4, 4, 6, 6, 7, 7, 7, 7, 8, 14, 15], np.uint8)
    assert np.array_equal(nvfp4.e2m1_encode(y), want)


def test_tensor_scale():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((2, 3, 40, 64)) * 3).astype(np.float16)
    amax = np.float32(np.abs(x.astype(np.float32)).max())
    assert nvfp4.tensor_scale(x) == np.float32(amax / np.float32(2688.0))
    assert nvfp4.tensor_scale(np.zeros((4, 64), np.float16)) == np.float32(1.0)


def test_hand_made_block_on_the_grid():
    # s_t = 1 and amax_b = 12: amax_b / 6 = 2 is an E4M3 value, so S_b = 2 and every
    # element that is twice a grid value round-trips exactly
    vals = np.array(MAGS * 2, np.float32) * 2.0
    vals[8:] *= -1
    x = vals.astype(np.float16).reshape(1, 16)
    codes, sb = nvfp4.quantize(x, np.float32(1.0))
    assert sb.tolist() == [[int(fp8.e4m3_encode(np.float32(2.0)))]]
    assert fp8.e4m3_decode(sb)[0] == 2.0
    assert np.array_equal(nvfp4.dequantize(codes, sb, 1.0), x.astype(np.float64))


def test_all_zero_block_and_negative_zero():
    x = np.zeros((2, 32), np.float16)
    x[1, :16] = -0.0
    codes, sb = nvfp4.quantize(x, np.float32(0.5))
    assert np.all(sb == 0) and np.all(codes == 0)
    assert np.all(nvfp4.dequantize(codes, sb, 0.5) == 0)


@pytest.mark.parametrize("mag", [1e-2, 1.0, 37.0, 900.0])
def test_block_max_lands_on_six(mag):
    rng = np.random.default_rng(int(mag * 10))
    x = (rng.standard_normal((64, 128)) * mag).astype(np.float16)
    s_t = nvfp4.tensor_scale(x)
    codes, sb = nvfp4.quantize(x, s_t)
    blocks = x.astype(np.float32).reshape(64, 8, 16)
    i = np.argmax(np.abs(blocks), axis=-1)
    c = np.take_along_axis(codes.reshape(64, 8, 16), i[..., None], axis=-1)[..., 0]
    S = fp8.e4m3_decode(sb)
    normal = S >= 2.0 ** -6          # a subnormal block scale has fewer bits: ratio bound below is for normal ones
    assert np.all((c[normal] & 7) == 7)


@pytest.mark.parametrize("mag", [1e-2, 1.0, 900.0])
def test_round_trip_error_bound(mag):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((32, 64)) * mag).astype(np.float16)
    s_t = nvfp4.tensor_scale(x)
    codes, sb = nvfp4.quantize(x, s_t)
    xh = nvfp4.dequantize(codes, sb, s_t)
    denom = (fp8.e4m3_decode(sb).astype(np.float64) * float(s_t))[:, :, None]
    err = np.abs(x.astype(np.float64).reshape(32, 4, 16) - xh.reshape(32, 4, 16))
    # half of the widest E2M1 gap (between 4 and 6) in units of the block's scale, plus the
    # rounding of the quotient fl32(x / fl32(S_b * s_t)) to float32
    assert np.all(err <= denom * (1.0 + 1e-6) + 1e-12)
    small = np.abs(xh.reshape(32, 4, 16)) < denom  # below 1: grid step 0.5
    assert np.all(err[small] <= denom[..., 0:1].repeat(16, -1)[small] * 0.25 * (1 + 1e-6) + 1e-12)


def test_e2m1_times_e4m3_is_an_exact_fp16_value():
    # the decode kernel forms fp16(e2m1 * S_b): every such product of finite codes is an fp16 value
    e2 = nvfp4.e2m1_decode(np.arange(16, dtype=np.uint8))
    e4 = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    e4 = e4[np.isfinite(e4)]
    prod = np.outer(e2, e4).ravel()
    assert np.array_equal(prod.astype(np.float16).astype(np.float64), prod)


# ---------------------------------------------------------------------------
# Pool layout: rebuild every m16n8k16 B tile the decode feeds to the tensor
# cores from the packed record by the PTX fragment description (B, ".col":
# b0 holds rows k = 2*tig, 2*tig + 1 and b1 rows k = 2*tig + 8, + 9 of column
# n = lane // 4), a different route from the packer's own loops.
# ---------------------------------------------------------------------------
from oracle import layout  # noqa: E402


def _stream_byte(rec, lane, p):
    return int(rec[((p // 16) * 32 + lane) * 16 + p % 16])


@pytest.mark.parametrize("d", [64, 128])
def test_key_record_fragments(d):
    rng = np.random.default_rng(d + 1)
    codes = rng.integers(0, 16, (16, d)).astype(np.uint8)
    scales = rng.integers(0, 256, (16, d // 16)).astype(np.uint8)
    rec = layout.nvfp4_pack_record(codes, scales, 0)
    ks_n = d // 16
    tile = np.full((16, d), -1)
    stile = np.full((16, ks_n), -1)
    for lane in range(32):
        g, tig = lane // 4, lane % 4
        for nt in range(2):
            for ks in range(ks_n):
                for r in range(2):  # b0 (r = 0) and b1 (r = 1): K rows 2tig + 8r, +1 = channels of k-step ks
                    byte = _stream_byte(rec, lane, (nt * ks_n + ks) * 2 + r)
                    tile[8 * nt + g, 16 * ks + 2 * tig + 8 * r] = byte & 15
                    tile[8 * nt + g, 16 * ks + 2 * tig + 8 * r + 1] = byte >> 4
                stile[8 * nt + g, ks] = rec[8 * d + g * 2 * ks_n + nt * ks_n + ks]
    assert np.array_equal(tile, codes) and np.array_equal(stile, scales)


@pytest.mark.parametrize("d", [64, 128])
def test_value_record_fragments(d):
    rng = np.random.default_rng(d + 2)
    codes = rng.integers(0, 16, (16, d)).astype(np.uint8)
    scales = rng.integers(0, 256, (16, d // 16)).astype(np.uint8)
    rec = layout.nvfp4_pack_record(codes, scales, 1)
    ks_n = d // 16
    tile = np.full((16, d), -1)
    stile = np.full((16, ks_n), -1)
    for lane in range(32):
        g, tig = lane // 4, lane % 4
        for nt in range(d // 8):
            for r in range(2):  # p.V: K = the 16 tokens, b0 rows 2tig, +1 (r = 0), b1 rows 2tig + 8, + 9
                byte = _stream_byte(rec, lane, nt * 2 + r)
                tile[2 * tig + 8 * r, 8 * nt + g] = byte & 15
                tile[2 * tig + 8 * r + 1, 8 * nt + g] = byte >> 4
        for r in range(2):
            for j in range(ks_n):
                for e in range(2):
                    stile[8 * r + 2 * tig + e, j] = rec[8 * d + ((tig * 2 + r) * ks_n + j) * 2 + e]
    assert np.array_equal(tile, codes) and np.array_equal(stile, scales)


def test_attention_over_nvfp4_values_matches_plain_dequantization():
    """The oracle attention reads keys and values through dequantize: check that
    softmax over e2m1 * S_b * s_t equals softmax over an explicit table lookup."""
    from oracle import attention
    rng = np.random.default_rng(5)
    k = (rng.standard_normal((40, 64)) * 2).astype(np.float16)
    q = rng.standard_normal(64).astype(np.float16)
    s_t = nvfp4.tensor_scale(k)
    codes, sb = nvfp4.quantize(k, s_t)
    table = {c: m for c, m in enumerate(MAGS + [-m for m in MAGS])}
    lookup = np.vectorize(table.get)(codes).astype(np.float64)
    kh = lookup * np.repeat(fp8.e4m3_decode(sb), 16, axis=1) * float(s_t)
    a = attention.softmax_attend(q, nvfp4.dequantize(codes, sb, s_t), kh, 0.125)
    b = attention.softmax_attend(q, kh, kh, 0.125)
    assert np.allclose(a, b, rtol=0, atol=0)
