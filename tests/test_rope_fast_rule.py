"""The single-precision shortcut of the RoPE rotation, checked on the CPU.

The append and the fused decode step compute each rotated value
RN_bf16(RN_f64(a*b + c*d)) (a, c bf16; b, d the fp32 table entries) in fp32
when an integer test on the bit patterns says that no bf16 rounding boundary
lies within the fp32 result's error bound, and by the exact double route
otherwise. This test restates that decision rule in numpy (fp32 products and
fma simulated exactly in wider precision) and checks, against the oracle's
own double-to-bf16 rounding, that every value the rule lets through rounds
to the same bf16 as the exact definition: on random values over 40 binades
and on inputs whose exact value lies within 4 fp32 ulps of a bf16 midpoint
or of a power of two. A failure here means the kernels' shortcut is unsound;
the GPU tests compare the kernels' bits with the oracle directly."""
import numpy as np

import oracle
from near_ties import near_tie_pairs


def _f32(x):
    return np.asarray(x, np.float64).astype(np.float32)


def _rule(a, b, c, d):
    """(bf16 bits of RN_bf16(s), accepted) for the kernel's fast path."""
    q = _f32(c * d)                                     # the product is exact in double
    qe = _f32(c * d - q.astype(np.float64))             # its rounding error, exact above underflow
    s = (np.longdouble(a * b) + np.longdouble(q.astype(np.float64))).astype(np.float32)  # one rounding
    S = s.view(np.uint32) & 0x7FFFFFFF
    Q = q.view(np.uint32) & 0x7FFFFFFF
    es, eq = (S >> 23).astype(np.int64), (Q >> 23).astype(np.int64)
    eqe = np.maximum(((qe.view(np.uint32) & 0x7FFFFFFF) >> 23).astype(np.int64), 1)
    L = (S & 0xFFFF).astype(np.int64)
    dist = np.minimum(np.minimum(np.abs(L - 0x8000), L + 0x4000), 0x18000 - L)
    k = eqe - es + 24
    need = np.where(k < 0, 2, np.where(k < 16, (1 << np.clip(k, 0, 15)) + 2, 0x20000))
    ok = (es >= 27) & (es <= 254) & ((Q == 0) | (eq >= 27)) & (dist >= need)
    u = s.view(np.uint32).astype(np.uint64)
    bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)  # round to nearest even
    return bits, ok


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
