"""Inputs for the append's near-tie tests.

The append rounds each rotated value RN_bf16(RN_f64(x1*c - x2*s)) (and
x2*c + x1*s for the second half of a head) once to bf16; a kernel may compute
it in single precision only where that provably gives the same bits. The
places where it could not are values whose exact rotation lies within a few
fp32 ulps of a bf16 rounding midpoint, or of a power of two (a binade edge,
where the bf16 and fp32 spacings change). This module finds bf16 pairs
(x1, x2) that land there for given table entries (c, s).

It only selects inputs. The expected outputs of every test that uses them
come from the oracle; the selection is itself checked with exact rational
arithmetic in a CPU test.
"""
from __future__ import annotations

import numpy as np

F32_PER_BF16 = 1 << 16  # fp32 ulps in one bf16 ulp


def offsets(r):
    """For double values r (nonzero, finite): (distance of |r| to the nearest
    bf16 rounding midpoint, distance of |r| to the nearest power of two), both
    in units of the fp32 ulp of |r|'s binade. Exact: frexp, ldexp and fmod
    do not round."""
    m, _ = np.frexp(np.abs(r))          # |r| = m * 2^e, m in [0.5, 1)
    u = np.ldexp(m, 24)                 # |r| in fp32 ulps of its binade, in [2^23, 2^24)
    low = np.fmod(u, float(F32_PER_BF16))
    d_mid = np.abs(low - F32_PER_BF16 / 2)
    d_edge = np.minimum(u - 2.0 ** 23, 2.0 ** 24 - u)
    return d_mid, d_edge


def _bf16_from_bits(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def random_bf16_bits(rng, n, emin=-30, emax=30):
    """n random bf16 patterns: random sign and 7-bit significand, exponent
    uniform in [emin, emax] (all normal numbers)."""
    sign = rng.integers(0, 2, size=n, dtype=np.uint32) << 15
    exp = (rng.integers(emin, emax + 1, size=n) + 127).astype(np.uint32) << 7
    man = rng.integers(0, 128, size=n, dtype=np.uint32)
    return (sign | exp | man).astype(np.uint16)


def _rot(x1, x2, c, s, half):
    # each product is exact in double (8-bit by 24-bit significands); the
    # sum rounds once, as in the append's definition
    return x1 * c - x2 * s if half == 0 else x2 * c + x1 * s


def near_tie_pairs(c, s, rng, n_samples=200_000, within=4.0, emin=-30, emax=30):
    """bf16 bit pairs (x1, x2) for one table entry (c, s) (fp32 values) whose
    rotated value, in either half, lies within `within` fp32 ulps of a bf16
    midpoint or of a power of two. Returns (x1_bits, x2_bits, kind) with kind
    0 = midpoint, 1 = binade edge.

    Midpoint cases come from random sampling (about 8 in 65,536 draws land
    within 4 ulps of a midpoint). Edge cases are aimed at: for powers of two
    t, x1 runs over the bf16 values around t / c and x2 over those around
    the solution of x1*c - x2*s = t (the second half likewise with the roles
    of x1 and x2 swapped). Two bf16 values of 8 significant bits rarely
    reach within 4 fp32 ulps of a power of two for a generic (c, s); they do
    where the angle is small (c near 1, s small), which the high-index
    table entries of every position supply."""
    c = float(c)
    s = float(s)
    import oracle
    out1, out2, kinds = [], [], []
    # -- midpoints, by sampling
    b1 = random_bf16_bits(rng, n_samples, emin, emax)
    b2 = random_bf16_bits(rng, n_samples, emin, emax)
    x1, x2 = _bf16_from_bits(b1), _bf16_from_bits(b2)
    for half in (0, 1):
        r = _rot(x1, x2, c, s, half)
        ok = (r != 0) & np.isfinite(r)
        d_mid, d_edge = offsets(np.where(ok, r, 1.0))
        hit = ok & ((d_mid <= within) | (d_edge <= within))
        out1.append(b1[hit]); out2.append(b2[hit])
        kinds.append(np.where(d_mid[hit] <= within, 0, 1))
    # -- binade edges, aimed at: for each power of two t (both signs), the
    # bf16 values around t / c for one element and, for each, the bf16
    # values around the other element that brings the rotation to t
    if s != 0.0 and c != 0.0:
        t = np.ldexp(1.0, np.arange(-12, 13))
        t = np.concatenate([t, -t])
        for half in (0, 1):
            base = oracle.f64_to_bf16(t / c).astype(np.int32)
            for j in range(-16, 17):
                bf = ((base + j) & 0xFFFF).astype(np.uint16)
                xf = _bf16_from_bits(bf)
                lead = xf * c                    # x1*c (half 0) or x2*c (half 1), exact
                # half 0: x1*c - x2*s = t -> x2 = (x1*c - t)/s; half 1: x2*c + x1*s = t -> x1 = (t - x2*c)/s
                other = (lead - t) / s if half == 0 else (t - lead) / s
                cand = oracle.f64_to_bf16(np.where(np.isfinite(other), other, 0.0)).astype(np.int32)
                for step in (-1, 0, 1):
                    bo = ((cand + step) & 0xFFFF).astype(np.uint16)
                    xo = _bf16_from_bits(bo)
                    good = np.isfinite(xf) & np.isfinite(xo) & ((bf & 0x7F80) != 0) & ((bo & 0x7F80) != 0)
                    a1, a2 = (xf, xo) if half == 0 else (xo, xf)
                    r = _rot(a1, a2, c, s, half)
                    good &= (r != 0) & np.isfinite(r)
                    _, d_edge = offsets(np.where(good, r, 1.0))
                    hit = good & (d_edge <= within)
                    p1, p2 = (bf, bo) if half == 0 else (bo, bf)
                    out1.append(p1[hit]); out2.append(p2[hit])
                    kinds.append(np.ones(int(hit.sum()), np.int64))
    return np.concatenate(out1), np.concatenate(out2), np.concatenate(kinds)


def near_tie_sets(table, positions, seed, **kw):
    """near_tie_pairs for every table entry i of every position:
    sets[k][i] = (x1_bits, x2_bits, kind) for positions[k]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [[near_tie_pairs(table[p, i, 0], table[p, i, 1], rng, **kw) for i in range(table.shape[1])]
            for p in positions]


def near_tie_rows(sets, positions, rows_per_position, heads, min_pairs=8):
    """Rows of bf16 head vectors [R][heads][d] (uint16 bits), R =
    rows_per_position * len(positions), row r at position
    positions[r // rows_per_position]: every rotation pair (i, i + d/2) of
    every head holds a near-tie pair for that position's table entry i
    (from near_tie_sets), distinct pairs first, then reused in turn.
    Returns (rows, row positions, distinct near-tie pairs placed, count of
    each kind placed)."""
    half = len(sets[0])
    R = rows_per_position * len(positions)
    rows = np.zeros((R, heads, 2 * half), np.uint16)
    pos = np.repeat(np.asarray(positions, np.int32), rows_per_position)
    distinct = 0
    kinds_placed = np.zeros(2, np.int64)
    need = rows_per_position * heads
    for k in range(len(positions)):
        for i in range(half):
            x1, x2, kind = sets[k][i]
            assert x1.size >= min_pairs, (positions[k], i, x1.size)
            take = np.arange(need) % x1.size
            distinct += min(need, x1.size)
            sl = slice(k * rows_per_position, (k + 1) * rows_per_position)
            rows[sl, :, i] = x1[take].reshape(rows_per_position, heads)
            rows[sl, :, i + half] = x2[take].reshape(rows_per_position, heads)
            kinds_placed += np.bincount(kind[take], minlength=2)
    return rows, pos, distinct, kinds_placed
