"""The single-precision shortcut of the RoPE rotation, checked on the CPU.

The append and the fused decode step compute each rotated value
RN_bf16(RN_f64(a*b + c*d)) (a, c bf16; b, d the fp32 table entries) in fp32
when both ends of the fp32 result's error interval round to the same bf16, and by the exact double route
otherwise. This test restates that decision rule in numpy (fp32 products and
fma simulated exactly in wider precision) and checks, against the oracle's
own double-to-bf16 rounding, that every value the rule lets through rounds
to the same bf16 as the exact definition (the rule: the fp32 result's error
interval, widened with directed rounding, rounds to one bf16 at both ends): on random values over 40 binades
and on inputs whose exact value lies within 4 fp32 ulps of a bf16 midpoint
or of a power of two. A failure here means the kernels' shortcut is unsound;
the GPU tests compare the kernels' bits with the oracle directly."""
import numpy as np

import oracle
from near_ties import near_tie_pairs


def _f32(x):
    return np.asarray(x, np.float64).astype(np.float32)


def _round_dir(x, up):
    """float32 nearest to the long double x in the given direction."""
    f = np.asarray(x, np.longdouble).astype(np.float32)
    fl = f.astype(np.longdouble)
    if up:
        return np.where(fl < x, np.nextafter(f, np.float32(np.inf)), f)
    return np.where(fl > x, np.nextafter(f, np.float32(-np.inf)), f)


def _bf16_rn(f):
    """bf16 bits of float32 values, round to nearest even (the hardware conversion)."""
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _rule(a, b, c, d):
    """(bf16 bits of RN_bf16(s), accepted) for the kernel's fast path."""
    q = _f32(c * d)                                     # the product is exact in double
    qe = _f32(c * d - q.astype(np.float64))             # its rounding error, exact above underflow
    s = (np.longdouble(a * b) + np.longdouble(q.astype(np.float64))).astype(np.float32)  # one rounding
    L = np.longdouble
    a_s = np.abs(s)
    t = _round_dir(np.abs(qe).astype(L) + L(2.0) ** -140, up=True)
    err = _round_dir(a_s.astype(L) * L(2.0) ** -24 + t.astype(L), up=True)
    lo = _round_dir(s.astype(L) - err.astype(L), up=False)
    hi = _round_dir(s.astype(L) + err.astype(L), up=True)
    ok = ((_bf16_rn(lo) == _bf16_rn(hi)) & (a_s >= np.float32(2.0 ** -100)) & (a_s < np.float32(2.0 ** 127)) &
          ((np.abs(q) >= np.float32(2.0 ** -100)) | (q == 0)))
    return _bf16_rn(s), ok


def _exact(a, b, c, d):
    x = np.longdouble(a) * np.longdouble(b) + np.longdouble(c) * np.longdouble(d)
    return oracle.f64_to_bf16(np.asarray(x, np.longdouble).astype(np.float64))


def _check(x1, x2, c, s):
    acc = 0
    for a, b, cc, dd in ((x1, c, -x2, s), (x2, c, x1, s)):   # both output halves
        bits, ok = _rule(a, b, cc, dd)
        ref = _exact(a, b, cc, dd)
        assert not np.any(ok & (bits != ref)), int(np.sum(ok & (bits != ref)))
        acc += int(ok.sum())
    return acc


def test_fast_rule_is_exact_on_random_values():
    assert np.finfo(np.longdouble).nmant >= 63, "needs an 80-bit long double to simulate the fma"
    rng = np.random.Generator(np.random.PCG64(11))
    tab = oracle.rope_table(1e6, 128, 4096)
    n = 2_000_000
    x1 = oracle.bf16_to_f64(oracle.f64_to_bf16(rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))))
    x2 = oracle.bf16_to_f64(oracle.f64_to_bf16(rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))))
    p, i = rng.integers(0, 4096, n), rng.integers(0, 64, n)
    accepted = _check(x1, x2, tab[p, i, 0].astype(np.float64), tab[p, i, 1].astype(np.float64))
    assert accepted > 0.999 * 2 * n  # the shortcut decides almost every value


def test_fast_rule_is_exact_at_near_ties():
    assert np.finfo(np.longdouble).nmant >= 63, "needs an 80-bit long double to simulate the fma"
    rng = np.random.Generator(np.random.PCG64(12))
    tab = oracle.rope_table(1e6, 128, 4096)
    seen = 0
    for p in (1, 100, 4095):
        for i in (0, 21, 42, 63):
            c, s = float(tab[p, i, 0]), float(tab[p, i, 1])
            b1, b2, _ = near_tie_pairs(c, s, rng, n_samples=60_000)
            x1 = (b1.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            x2 = (b2.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            _check(x1, x2, np.full_like(x1, c), np.full_like(x1, s))
            seen += x1.size
    assert seen > 1000
