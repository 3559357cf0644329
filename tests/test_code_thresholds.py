"""The 2-bit codes of the KIVI quantize kernel come from three fp16 thresholds
per channel (keys) or token (values) instead of a division per element. This
checks the derivation those thresholds follow, written out here with exact
rational arithmetic, against the oracle's group formula (oracle.kivi) on every
fp16 value of many group ranges:

* code >= k  <=>  fl32(x - z) >= D_k, with D_2 = RU32(s (1.5 - 2^-24)) and
  D_1, D_3 the smallest fp32 above s (0.5 + 2^-25), s (2.5 + 2^-23): the tie
  rules of rint (half to even) and of the fp32 quotient (m = k - 1/2 has an
  even significand);
* theta_k = the smallest fp16 x with fl32(x - z) >= D_k: RU16(z + D_k) where
  that candidate and the fp16 value below it confirm it, else a bisection.

The GPU kernel is checked against the oracle byte for byte by the GPU tests;
this test pins the arithmetic argument itself, on the CPU.
"""
from fractions import Fraction as Fr

import numpy as np

from oracle import kivi


def _rnd32(fr, up):
    """The float32 next to the rational fr, rounded up (up) or down."""
    x = np.float32(float(fr))
    if up:
        while Fr(float(x)) < fr:
            x = np.nextafter(x, np.float32(np.inf))
        while Fr(float(np.nextafter(x, np.float32(-np.inf)))) >= fr:
            x = np.nextafter(x, np.float32(-np.inf))
    else:
        while Fr(float(x)) > fr:
            x = np.nextafter(x, np.float32(-np.inf))
        while Fr(float(np.nextafter(x, np.float32(np.inf)))) <= fr:
            x = np.nextafter(x, np.float32(np.inf))
    return x


def _step(s, k):
    """D_k: the smallest float32 d with rint(fl32(d / s)) >= k (s > 0)."""
    s = Fr(float(s))
    m = Fr(2 * k - 1, 2)
    if k == 2:
        return _rnd32(m * s - Fr(1, 2 ** 24) * s, up=True)
    h = Fr(1, 2 ** 25) if k == 1 else Fr(1, 2 ** 23)
    up, dn = _rnd32(m * s + h * s, True), _rnd32(m * s + h * s, False)
    return np.nextafter(up, np.float32(np.inf)) if up == dn else up


def _key(b):
    b = int(b)
    return -(b & 0x7FFF) if b & 0x8000 else (b & 0x7FFF)


def _bits(key):
    return key if key >= 0 else (0x8000 | -key)


def _half(b):
    return np.array([b], np.uint16).view(np.float16)[0]


def _threshold(z, s, k):
    """theta_k as fp16 bits (0x7C00 when s = 0: every code is 0)."""
    if np.float32(s) == 0:
        return 0x7C00
    d = _step(s, k)
    reaches = lambda key: np.float32(np.float32(_half(_bits(key))) - np.float32(z)) >= d
    t = _rnd32(Fr(float(np.float32(z))) + Fr(float(d)), up=True)
    x0 = np.float16(t)
    if np.float32(x0) < t:
        x0 = np.nextafter(x0, np.float16(np.inf))
    k0 = _key(np.array([x0], np.float16).view(np.uint16)[0])
    kz = _key(np.array([z], np.float16).view(np.uint16)[0])
    r0 = reaches(k0)
    r1 = k0 - 1 > kz and reaches(k0 - 1)
    if r0 and not r1:
        return _bits(k0)
    lo, hi = (kz, k0 - 1) if r0 else (k0, 0x7C00)
    for _ in range(17):
        if hi - lo <= 1:
            break
        mid = lo + (hi - lo) // 2
        if reaches(mid):
            hi = mid
        else:
            lo = mid
    return _bits(hi)


def _ranges():
    rng = np.random.default_rng(17)
    fixed = [(-3, 3), (-1000, 1000), (-65504, 65504), (-1e-7, 1e-7), (-2, 0), (0, 2), (-6e-8, 6e-8), (1, 1),
             (0, 0), (-5e4, 3e-5), (-3e-5, 5e4), (-1000, 1e-3), (100, 100.5), (-60000, 2), (-2, 60000),
             (5e-5, 7e-5), (-0.75, 0.25), (0.0, 65504), (1e-7, 3e-7)]
    rand = [tuple(sorted(rng.standard_normal(2) * 10 ** rng.uniform(-7, 4.5))) for _ in range(60)]
    return fixed + rand


def test_thresholds_reproduce_the_group_formula_on_every_fp16_value():
    for a, b in _ranges():
        mn, mx = np.float16(a), np.float16(b)
        if mn > mx:
            mn, mx = mx, mn
        keys = np.arange(_key(np.array([mn], np.float16).view(np.uint16)[0]),
                         _key(np.array([mx], np.float16).view(np.uint16)[0]) + 1)
        xs = np.where(keys >= 0, keys, 0x8000 | (-keys)).astype(np.uint16).view(np.float16)
        # the oracle's codes of every x in [mn, mx], each in a group whose min and max are mn and mx
        rows = np.stack([np.full(xs.size, mn), np.full(xs.size, mx), xs], axis=-1).astype(np.float16)
        codes, s16, z16 = kivi.quantize_groups(rows, 2)
        want = codes[:, 2].astype(int)
        s, z = s16[0], z16[0]
        th = [_half(_threshold(z, s, k)) for k in (1, 2, 3)]
        got = sum((xs >= t).astype(int) for t in th)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (a, b, float(z), float(s), [float(t) for t in th], xs[bad[:4]])


def test_a_step_near_zero_moves_by_the_rounding_of_x_minus_z():
    """Range [-3, 3]: s = 2, the step to code 2 sits near x = 0, where fl32(x + 3)
    rounds; it lands on a tiny negative fp16 value, not on 0 (the candidate
    RU16(z + D_2) = 0 is rejected and the bisection finds it)."""
    z, s = np.float16(-3.0), np.float16(2.0)
    t2 = _half(_threshold(z, s, 2))
    assert float(t2) < 0 and abs(float(t2)) < 1e-6
    rows = np.array([[-3, 3, t2], [-3, 3, np.nextafter(t2, np.float16(-np.inf))]], np.float16)
    codes = kivi.quantize_groups(rows, 2)[0][:, 2]
    assert codes.tolist() == [2, 1]
