"""Pins of the byte accounting against the worked numbers printed on the pages."""
import os
from fractions import Fraction

import pytest

from oracle import sizes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [c.strip() for c in line.split("|")]


@pytest.mark.parametrize("row", list(_rows("kv_bytes.txt")), ids=lambda r: r[0])
def test_kv_bytes_worked_numbers(row):
    _, layers, batch, seq, heads, dim, bpe, expected = row
    got = sizes.kv_cache_bytes(int(layers), int(batch), int(seq), int(heads), int(dim), Fraction(bpe))
    assert got == int(expected)


def test_page_rounded_values():
    gib = 2 ** 30
    # "约 2GiB ... 约 64GiB" and "约 0.5GiB" are exact binary multiples at these shapes
    assert sizes.kv_cache_bytes(32, 1, 4096, 32, 128, 2) / gib == 2
    assert sizes.kv_cache_bytes(32, 1, 32768, 1, 128, 2) / gib == Fraction(1, 2)
    assert sizes.kv_cache_bytes(32, 1, 1, 32, 128, 2) / 1024 == 512


def test_worked_ratios():
    rows = {r[0]: r for r in _rows("kv_ratios.txt")}
    ab = sizes.average_bits(8064, 4, 128, 16)
    assert ab == Fraction(rows["avg_bits"][2])
    assert round(float(ab), 2) == float(rows["avg_bits"][3])
    ov = sizes.metadata_overhead(64, 4, 2, 1)
    assert ov == Fraction(rows["meta_overhead"][2])
    assert round(float(ov), 3) == float(rows["meta_overhead"][3])
    assert sizes.kv_elements_per_token(32, 32, 128) == int(rows["elems_per_token"][2])


def test_fp8_halves_fp16_bytes():
    # FP8 stores one byte per element, FP16 two (section 5 of the aiinfraguide page)
    for s in (1, 4096, 32768):
        assert sizes.kv_cache_bytes(1, 64, s, 8, 128, 1) * 2 == sizes.kv_cache_bytes(1, 64, s, 8, 128, 2)


def test_kivi_layout_bytes():
    # 2-bit, D = 128: 32 B key codes + 16 B key meta + 32 B value codes + 4 B value meta per token-head
    assert sizes.kivi_bytes_per_grouped_token(128, 2, 2) == 84
    assert sizes.kivi_bytes_per_grouped_token(128, 4, 4) == 148
    # the codes alone are 16/bits times smaller than fp16 (8x at 2 bits, the aiinfraguide
    # page's section 4); metadata brings the 2-bit ratio to 512/84 ~ 6.1x per grouped token
    g = sizes.kivi_group_bytes(128, 2, 2)
    assert g["k_codes"] * 8 == 32 * 128 * 2
    assert (g["k_codes"] + g["v_codes"]) * 8 == sizes.kv_cache_bytes(1, 1, 32, 1, 128, 2)
    assert 6 < Fraction(512, sizes.kivi_bytes_per_grouped_token(128, 2, 2)) < 6.2
    b = sizes.kivi_buffer_bytes(4, 8, 128, 2, 2, 128, 131584)
    assert b["k_codes"] == 4 * 8 * (131584 // 32) * 1024
    assert b["k_res"] == 4 * 8 * 128 * 128 * 2


def test_decode_bytes_stream_case():
    # 128K streaming case: 130944 grouped + 128 residual tokens, 4 x 8 kv heads, 64 q heads
    n = sizes.decode_bytes_kivi(4, 8, 64, 128, 2, 2, 130944, 128)
    assert n == 84 * 130944 * 32 + 128 * 512 * 32 + 2 * 4 * 64 * 128 * 2
