"""The near-tie input selection (tests/near_ties.py) against exact rational
arithmetic: every pair it returns has an exact rotated value within the
stated fp32-ulp distance of a bf16 rounding midpoint or of a power of two.
CPU only; the GPU append tests rely on this selection."""
from fractions import Fraction

import numpy as np

import oracle
from near_ties import near_tie_pairs, near_tie_rows, near_tie_sets


def _exact_distances(r):
    """(|r| to the nearest bf16 midpoint, |r| to the nearest power of two),
    in fp32 ulps of |r|'s binade, for a nonzero rational r."""
    a = abs(r)
    e = 0
    while a >= 2 ** (e + 1):
        e += 1
    while a < 2 ** e:
        e -= 1
    ulp32 = Fraction(2) ** (e - 23)
    ulp16 = Fraction(2) ** (e - 7)
    k = a // ulp16
    mid = (k + Fraction(1, 2)) * ulp16
    d_mid = min(abs(a - mid), abs(a - (mid - ulp16)), abs(a - (mid + ulp16))) / ulp32
    d_edge = min(a - Fraction(2) ** e, Fraction(2) ** (e + 1) - a) / ulp32
    return d_mid, d_edge


def _f(bits16):
    return Fraction(float(np.array([int(bits16) << 16], np.uint32).view(np.float32)[0]))


def test_selected_pairs_are_near_ties_exactly():
    tab = oracle.rope_table(1e6, 128, 4096)
    rng = np.random.Generator(np.random.PCG64(7))
    seen = np.zeros(2, int)
    for p, i in ((1, 0), (100, 10), (4095, 63), (17, 40)):
        c, s = tab[p, i, 0], tab[p, i, 1]
        x1, x2, kind = near_tie_pairs(c, s, rng, n_samples=100_000)
        assert x1.size > 0
        cf, sf = Fraction(float(c)), Fraction(float(s))
        for j in np.linspace(0, x1.size - 1, min(40, x1.size)).astype(int):
            a, b = _f(x1[j]), _f(x2[j])
            best = None
            for r in (a * cf - b * sf, b * cf + a * sf):
                if r == 0:
                    continue
                dm, de = _exact_distances(r)
                v = dm if kind[j] == 0 else de
                best = v if best is None or v < best else best
            # the selection works on the sum rounded to double: 2^-29 fp32 ulps of slack
            assert best is not None and best <= Fraction(4) + Fraction(1, 1 << 20), (p, i, j, float(best))
            seen[kind[j]] += 1
    assert seen[0] > 0 and seen[1] > 0


def test_rows_fill_every_pair_with_a_near_tie():
    tab = oracle.rope_table(1e6, 64, 64)
    sets = near_tie_sets(tab, [3, 40], seed=5, n_samples=100_000)
    rows, pos, distinct, kinds = near_tie_rows(sets, [3, 40], 1, 3, min_pairs=1)
    assert rows.shape == (2, 3, 64) and list(pos) == [3, 40]
    assert distinct > 0 and kinds.sum() == 2 * 3 * 32
    assert np.all((rows & 0x7F80) != 0)  # normal numbers only
