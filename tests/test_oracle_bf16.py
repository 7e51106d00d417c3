"""Pins for the oracle's bf16 conversions against the number-format definition.

double -> bf16 is checked against brute force: the two bf16 neighbours of the
exact value (found by bisection over all finite bf16 values) and an exact
rational comparison of the distances, ties to the even pattern, overflow to
infinity past the halfway point above the largest finite value.
"""
import bisect
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _bits_to_float(h):
    return struct.unpack("<f", struct.pack("<I", (h & 0xFFFF) << 16))[0]


def _positive_table():
    pats = [h for h in range(0x0000, 0x7F80)]  # +0 .. largest finite
    vals = [_bits_to_float(h) for h in pats]
    return pats, vals


PATS, VALS = _positive_table()


def brute_bf16(x: float) -> int:
    if math.isnan(x):
        return 0xFFC0 if math.copysign(1.0, x) < 0 else 0x7FC0
    sgn = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if math.isinf(a):
        return sgn | 0x7F80
    i = bisect.bisect_left(VALS, a)
    if i < len(VALS) and VALS[i] == a:
        return sgn | PATS[i]
    if i == len(VALS):  # above the largest finite value
        lo_pat, lo = PATS[-1], Fraction(VALS[-1])
        hi_pat, hi = 0x7F80, Fraction(2) ** 128  # the next step of an unbounded exponent
    else:
        lo_pat, lo = PATS[i - 1], Fraction(VALS[i - 1])
        hi_pat, hi = PATS[i], Fraction(VALS[i])
    fa = Fraction(a)
    dl, dh = fa - lo, hi - fa
    if dl < dh:
        pick = lo_pat
    elif dh < dl:
        pick = hi_pat
    else:
        pick = lo_pat if lo_pat % 2 == 0 else hi_pat
    return sgn | pick


def test_roundtrip_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    d = oracle.bf16_to_f64(h)
    # bf16 -> double against numpy's float32 view of the shifted bits
    with np.errstate(invalid="ignore"):  # signalling NaN patterns widen to quiet NaNs
        ref = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    finite = ~np.isnan(ref)
    assert np.array_equal(d[finite], ref[finite])
    assert np.all(np.isnan(d[~finite]))
    back = oracle.f64_to_bf16(d)
    assert np.array_equal(back[finite], h[finite])
    # NaNs come back as the canonical quiet NaN with the sign kept
    nan_h = h[~finite]
    assert np.all((back[~finite] & 0x7FFF) == 0x7FC0)
    assert np.array_equal(back[~finite] & 0x8000, nan_h & 0x8000)


def _edge_values():
    xs = [0.0, -0.0, 1.0, -1.0, math.inf, -math.inf, 1e-300, -1e-300, 5e-324,
          2.0 ** -133, 2.0 ** -134, 2.0 ** -134 * (1 + 2 ** -52), 2.0 ** -135,
          2.0 ** -126, 2.0 ** -126 * (1 - 2 ** -9), 2.0 ** -127 * 3,
          float.fromhex("0x1.fep127"), float.fromhex("0x1.fefffffffffffp127"),
          float.fromhex("0x1.ff00000000000p127"), float.fromhex("0x1.ff00000000001p127"),
          2.0 ** 128, 1e300, -1e300]
    # exact halfway points between consecutive bf16 values, and one double ulp either side
    for h in (0x3F80, 0x3F81, 0x4000, 0x0001, 0x0002, 0x007F, 0x0080, 0x7F7E, 0x1234, 0x4B00):
        lo, hi = _bits_to_float(h), _bits_to_float(h + 1)
        mid = (lo + hi) / 2.0  # exact in double
        xs += [mid, -mid, math.nextafter(mid, math.inf), math.nextafter(mid, -math.inf)]
    # values that a detour through float32 would round twice
    xs += [1.0 + 2 ** -8 + 2 ** -30, 1.0 + 2 ** -8 - 2 ** -30, 1.0 + 3 * 2 ** -9 + 2 ** -40]
    return xs


def test_edge_cases_against_brute_force():
    for x in _edge_values():
        assert oracle.bf16_from_double_scalar(x) == brute_bf16(x), x


def test_random_doubles_against_brute_force():
    r = np.random.Generator(np.random.PCG64(7))
    xs = np.concatenate([
        r.standard_normal(4000),
        r.standard_normal(2000) * 1e-38,
        r.standard_normal(1000) * 1e-40,
        r.standard_normal(1000) * 3e38,
        np.ldexp(r.uniform(1, 2, 2000), r.integers(-140, 130, 2000)) * r.choice([-1, 1], 2000),
    ])
    got = oracle.f64_to_bf16(xs)
    for x, g in zip(xs.tolist(), got.tolist()):
        assert g == brute_bf16(x), (x, hex(g), hex(brute_bf16(x)))


def test_double_rounding_is_avoided():
    # 1 + 2^-8 + tiny lies just above the bf16 halfway point 1 + 2^-8; a
    # conversion through float32 would first land exactly on the halfway point
    # and then round to even (down). One rounding goes up.
    x = 1.0 + 2 ** -8 + 2 ** -40
    assert oracle.bf16_from_double_scalar(x) == 0x3F81
    assert oracle.bf16_from_double_scalar(1.0 + 2 ** -8) == 0x3F80  # exact tie -> even
    assert oracle.bf16_from_double_scalar(1.0 + 3 * 2 ** -8) == 0x3F82  # tie -> even (up)
