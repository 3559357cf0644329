"""Pins of the packed-cache layout.

The packer in ``oracle.layout`` is checked against the mma.sync m16n8k16
operand-fragment semantics of the PTX ISA (B operand, ``.col``: register b0
holds rows ``k = 2*tig + {0,1}`` and b1 rows ``k = 2*tig + 8 + {0,1}`` of
column ``n = lane // 4``), combined with the documented field-extraction rule:
each 16-bit half of an extracted register is an fp16 subnormal whose value is
``code * 2^(P - 24)``. This is a different route to the same bytes than the
packer's own loops, so an index slip in either shows up here.
"""
import numpy as np
import pytest

from oracle import kivi, layout

# field extraction rule of the decode kernel: an operation on the 32-bit word
# (a shift, or a swap of the two bytes of each 16-bit half), then a mask that
# keeps bits [P, P + bits) of each half; returns (operation, P). For 2 bits the
# B operand of n-tile nt%4 takes: 0 -> (w << 4, w >> 4) at P = 6, 1 -> the same
# at P = 8, 2 -> (w, swap(w)) at P = 6, 3 -> the same at P = 8 (b0, b1 = r 0, 1).
def _extract_rule(bits, r, nt):
    if bits == 2:
        op = [("shl", 4), ("shr", 4), ("shl", 0), ("swap", 0)][2 * ((nt % 4) // 2) + r]
        p = 6 if nt % 2 == 0 else 8
    else:
        op = [("shl", 6), ("shl", 2), ("shr", 2), ("shr", 6)][nt % 4]
        p = 6
    return op, p


def _extract(word, bits, r, nt):
    (kind, n), p = _extract_rule(bits, r, nt)
    w = int(word)
    if kind == "shl":
        w = (w << n) & 0xFFFFFFFF
    elif kind == "shr":
        w = w >> n
    else:
        w = ((w & 0x00FF00FF) << 8) | ((w >> 8) & 0x00FF00FF)
    mask = ((1 << bits) - 1) << p
    w &= mask | (mask << 16)
    lo = np.uint16(w & 0xFFFF).view(np.float16)
    hi = np.uint16(w >> 16).view(np.float16)
    scale = 2.0 ** (24 - p)
    return float(lo) * scale, float(hi) * scale


def _word(packed_u32, lane, u):
    return packed_u32[(u // 4) * 128 + lane * 4 + u % 4]


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("d", [64, 128])
def test_key_fragments(bits, d):
    rng = np.random.default_rng(bits * 1000 + d)
    codes = rng.integers(0, 2 ** bits, size=(32, d), dtype=np.uint8)
    words = layout.pack_key_codes(codes, bits).view(np.uint32)
    assert words.size * 4 == 32 * d * bits // 8
    # rebuild every B tile of q . k^T: K = 16 channels of k-step ks, N = 8 tokens of n-tile nt
    for ks in range(d // 16):
        for nt in range(4):
            tile = np.full((16, 8), -1.0)
            for lane in range(32):
                g, tig = lane // 4, lane % 4
                for r in range(2):
                    u = ks if bits == 2 else 2 * ks + r
                    lo, hi = _extract(_word(words, lane, u), bits, r, nt)
                    tile[2 * tig + 8 * r, g] = lo
                    tile[2 * tig + 8 * r + 1, g] = hi
            want = codes[8 * nt:8 * nt + 8, 16 * ks:16 * ks + 16].T.astype(np.float64)
            assert np.array_equal(tile, want), (ks, nt)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("d", [64, 128])
def test_value_fragments(bits, d):
    rng = np.random.default_rng(bits * 7 + d)
    codes = rng.integers(0, 2 ** bits, size=(32, d), dtype=np.uint8)
    words = layout.pack_value_codes(codes, bits).view(np.uint32)
    nq = d // 32
    # B tiles of p . V: K = 16 tokens of k-step ks, N = 8 channels of n-tile nt
    for ks in range(2):
        for nt in range(d // 8):
            tile = np.full((16, 8), -1.0)
            for lane in range(32):
                g, tig = lane // 4, lane % 4
                for r in range(2):
                    u = ks * nq + nt // 4 if bits == 2 else (2 * ks + r) * nq + nt // 4
                    lo, hi = _extract(_word(words, lane, u), bits, r, nt)
                    tile[2 * tig + 8 * r, g] = lo
                    tile[2 * tig + 8 * r + 1, g] = hi
            want = codes[16 * ks:16 * ks + 16, 8 * nt:8 * nt + 8].astype(np.float64)
            assert np.array_equal(tile, want), (ks, nt)


def test_simulated_scores_match_plain_product():
    """q'.codes through the fragments equals the plain matrix product."""
    rng = np.random.default_rng(11)
    d = 128
    codes = rng.integers(0, 4, size=(32, d), dtype=np.uint8)
    words = layout.pack_key_codes(codes, 2).view(np.uint32)
    qp = rng.standard_normal(d)
    scores = np.zeros(32)
    for ks in range(d // 16):
        for nt in range(4):
            for lane in range(32):
                g, tig = lane // 4, lane % 4
                lo, hi = _extract(_word(words, lane, ks), 2, 0, nt)
                lo2, hi2 = _extract(_word(words, lane, ks), 2, 1, nt)
                c = 16 * ks + 2 * tig
                scores[8 * nt + g] += qp[c] * lo + qp[c + 1] * hi + qp[c + 8] * lo2 + qp[c + 9] * hi2
    assert np.allclose(scores, codes.astype(np.float64) @ qp, rtol=1e-12, atol=1e-12)


def test_meta_records():
    rng = np.random.default_rng(12)
    d = 128
    s = rng.standard_normal(d).astype(np.float16)
    z = rng.standard_normal(d).astype(np.float16)
    m = layout.pack_key_meta(s, z).view(np.float16).reshape(d // 16, 4, 8)
    for ks in range(d // 16):
        for tig in range(4):
            d0 = 16 * ks + 2 * tig
            assert np.array_equal(m[ks, tig, :4], s[[d0, d0 + 1, d0 + 8, d0 + 9]])
            assert np.array_equal(m[ks, tig, 4:], z[[d0, d0 + 1, d0 + 8, d0 + 9]])
    vs = rng.standard_normal(32).astype(np.float16)
    vz = rng.standard_normal(32).astype(np.float16)
    vm = layout.pack_value_meta(vs, vz).view(np.float16).reshape(2, 4, 8)
    for tig in range(4):
        toks = [8 * nt + 2 * tig + j for nt in range(4) for j in range(2)]
        assert np.array_equal(vm[0, tig], vs[toks]) and np.array_equal(vm[1, tig], vz[toks])


def test_pack_cache_shapes():
    rng = np.random.default_rng(13)
    c = kivi.KiviCache(2, 3, 64, 2, 4, 128)
    k = (rng.standard_normal((2, 3, 300, 64))).astype(np.float16)
    c.prefill(k, k)
    p = layout.pack_cache(c)
    ng = c.n_grouped // 32
    assert p["k_codes"].shape == (2, 3, ng, 512)
    assert p["v_codes"].shape == (2, 3, ng, 1024)
    assert p["k_meta"].shape == (2, 3, ng, 256)
    assert p["v_meta"].shape == (2, 3, ng, 128)


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_block_order_fragments(d):
    """The FP8 in-block order against the m16n8k16 B-fragment description:
    keys give B[k = channel][n = token] tiles, values B[k = token][n = channel]."""
    rng = np.random.default_rng(d)
    blk = rng.integers(0, 256, size=(1, 1, 16, d), dtype=np.uint8)
    for vl in (0, 1):
        perm = layout.fp8_block_order(d, vl)
        assert sorted(perm) == list(range(16 * d))          # a permutation
        packed = layout.fp8_pack_pool(blk, vl)[0, 0]
        lane_bytes = lambda lane: np.array([packed[((p // 16) * 32 + lane) * 16 + p % 16] for p in range(d // 2)])
        nat = blk[0, 0]
        if vl == 0:
            for nt in range(2):
                for ks in range(d // 16):
                    tile = np.zeros((16, 8), np.int64)
                    for lane in range(32):
                        g, tig = lane // 4, lane % 4
                        lb = lane_bytes(lane)
                        i0 = (nt * (d // 16) + ks) * 2
                        tile[2 * tig, g], tile[2 * tig + 1, g] = lb[2 * i0], lb[2 * i0 + 1]
                        tile[2 * tig + 8, g], tile[2 * tig + 9, g] = lb[2 * i0 + 2], lb[2 * i0 + 3]
                    assert np.array_equal(tile, nat[8 * nt:8 * nt + 8, 16 * ks:16 * ks + 16].T)
        else:
            for nt in range(d // 8):
                tile = np.zeros((16, 8), np.int64)
                for lane in range(32):
                    g, tig = lane // 4, lane % 4
                    lb = lane_bytes(lane)
                    tile[2 * tig, g], tile[2 * tig + 1, g] = lb[4 * nt], lb[4 * nt + 1]
                    tile[2 * tig + 8, g], tile[2 * tig + 9, g] = lb[4 * nt + 2], lb[4 * nt + 3]
                assert np.array_equal(tile, nat[:, 8 * nt:8 * nt + 8])
        assert np.array_equal(layout.fp8_unpack_pool(layout.fp8_pack_pool(blk, vl), d, vl), blk)


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_key_order_for_fp8_tensor_cores(d):
    """value_layout 2 against the m16n8k32 8-bit operand fragments: lane (g, tig)
    holds B[k][n] for k = 4*tig .. 4*tig + 3 (first register) and 16 + 4*tig ..
    (second), n = g, with k = channel and n = token; a simulated m16n8k32 over
    those fragments and row-major query bytes gives the plain product."""
    rng = np.random.default_rng(d + 2)
    blk = rng.integers(0, 256, size=(1, 1, 16, d), dtype=np.uint8)
    perm = layout.fp8_block_order(d, 2)
    assert sorted(perm) == list(range(16 * d))
    packed = layout.fp8_pack_pool(blk, 2)[0, 0]
    assert np.array_equal(layout.fp8_unpack_pool(layout.fp8_pack_pool(blk, 2), d, 2), blk)
    lane_bytes = lambda lane: np.array([packed[((p // 16) * 32 + lane) * 16 + p % 16] for p in range(d // 2)])
    nat = blk[0, 0].astype(np.int64)
    qa = rng.integers(-8, 8, size=(16, d))            # a query tile (rows = heads), small integers
    for nt in range(2):
        acc = np.zeros((16, 8), np.int64)
        for kk in range(d // 32):
            tile = np.zeros((32, 8), np.int64)
            for lane in range(32):
                g, tig = lane // 4, lane % 4
                lb = lane_bytes(lane)
                w0 = (nt * (d // 32) + kk) * 2
                tile[4 * tig:4 * tig + 4, g] = lb[4 * w0:4 * w0 + 4]
                tile[16 + 4 * tig:16 + 4 * tig + 4, g] = lb[4 * w0 + 4:4 * w0 + 8]
            assert np.array_equal(tile, nat[8 * nt:8 * nt + 8, 32 * kk:32 * kk + 32].T)
            # A fragment of m16n8k32: rows g / g + 8, columns 4*tig.. and 16 + 4*tig.. of the tile
            a = np.zeros((16, 32), np.int64)
            for lane in range(32):
                g, tig = lane // 4, lane % 4
                for r in (g, g + 8):
                    for half in (0, 16):
                        cols = slice(half + 4 * tig, half + 4 * tig + 4)
                        a[r, cols] = qa[r, 32 * kk:32 * kk + 32][cols]
            acc += a @ tile
        assert np.array_equal(acc, qa @ nat[8 * nt:8 * nt + 8].T)
