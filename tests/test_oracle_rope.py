"""Pins for the oracle's RoPE table and rotation (rotate-half pairing).

Checked against: an independent high-precision evaluation of every table entry
(mpmath, 50 digits), closed forms (position 0, the frequency-1 and
frequency-1e-3 columns at theta = 1e6, d = 128), and the properties that define
a rotary embedding: norm preservation, invertibility, and dot products that
depend only on the position difference.
"""
import math

import numpy as np
import pytest

import oracle
from workloads import bf16_normal


def test_table_position_zero_is_identity():
    t = oracle.rope_table(1e6, 128, 4)
    assert np.all(t[0, :, 0] == 1.0) and np.all(t[0, :, 1] == 0.0)


def test_table_closed_form_columns():
    # theta^(-2i/d) is 1 for i = 0 and theta^(-1/2) = 1e-3 for i = d/4
    t = oracle.rope_table(1e6, 128, 3001)
    for p in (1, 2, 3, 17, 1000, 3000):
        assert t[p, 0, 0] == np.float32(math.cos(p)) and t[p, 0, 1] == np.float32(math.sin(p))
        ang = p / 1000.0
        assert abs(float(t[p, 32, 0]) - math.cos(ang)) <= 2 ** -24
        assert abs(float(t[p, 32, 1]) - math.sin(ang)) <= 2 ** -24
    # cos(1) and sin(1) printed to 16 digits
    assert abs(float(t[1000, 32, 0]) - 0.5403023058681398) <= 2 ** -24
    assert abs(float(t[1000, 32, 1]) - 0.8414709848078965) <= 2 ** -24


@pytest.mark.parametrize("d,theta", [(64, 1e6), (128, 1e6), (128, 1e4)])
def test_table_against_high_precision(d, theta):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    positions = [0, 1, 2, 15, 16, 17, 255, 1024, 8191, 32767]
    t = oracle.rope_table(theta, d, max(positions) + 1)
    for p in positions:
        for i in range(d // 2):
            ang = mpmath.mpf(p) * mpmath.power(mpmath.mpf(theta), -mpmath.mpf(2 * i) / d)
            for j, f in ((0, mpmath.cos), (1, mpmath.sin)):
                exact = float(f(ang))
                got = float(t[p, i, j])
                # fp32 rounding of a double within a few double ulps of the truth
                ulp = np.spacing(np.float32(abs(exact))) if exact != 0 else 2 ** -149
                assert abs(got - exact) <= 0.5 * ulp * (1 + 1e-6) + 1e-15 * max(1.0, p), (p, i, j)


def _rot_f64(x, table, p):
    """Rotation applied to float64 values (no rounding), for property checks."""
    d = x.shape[-1]
    h = d // 2
    c = table[p, :, 0].astype(np.float64)
    s = table[p, :, 1].astype(np.float64)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def test_rotate_position_zero_is_bit_exact_copy():
    r = np.random.Generator(np.random.PCG64(3))
    x = bf16_normal(r, (5, 128))
    t = oracle.rope_table(1e6, 128, 2)
    assert np.array_equal(oracle.rope_rotate(x, t, 0), x)


def test_rotate_is_single_rounding_of_exact_rotation():
    # the exact rotation in double (products of bf16 and fp32 values are exact)
    # rounded once to bf16 must equal the oracle
    r = np.random.Generator(np.random.PCG64(4))
    x = bf16_normal(r, (16, 64))
    t = oracle.rope_table(1e6, 64, 100)
    for p in (1, 5, 99):
        y = oracle.rope_rotate(x, t, p)
        exact = _rot_f64(oracle.bf16_to_f64(x), t, p)
        assert np.array_equal(y, oracle.f64_to_bf16(exact))


def test_rotate_pairing_is_rotate_half():
    # a unit vector in coordinate i moves into coordinate i + d/2 (not i + 1)
    d = 8
    t = oracle.rope_table(10.0, d, 4)
    x = np.zeros((1, d), np.uint16)
    x[0, 1] = 0x3F80  # 1.0 at i = 1
    y = oracle.bf16_to_f64(oracle.rope_rotate(x, t, 3))[0]
    ang = 3 * 10.0 ** (-2 * 1 / d)
    assert abs(y[1] - math.cos(ang)) < 1e-2 and abs(y[1 + d // 2] - math.sin(ang)) < 1e-2
    assert np.count_nonzero(y) == 2


def test_rotate_preserves_norm_and_inverts():
    r = np.random.Generator(np.random.PCG64(5))
    x = bf16_normal(r, (64, 128))
    t = oracle.rope_table(1e6, 128, 9000)
    xf = oracle.bf16_to_f64(x)
    for p in (1, 7, 512, 8191, 8999):
        y = oracle.bf16_to_f64(oracle.rope_rotate(x, t, p))
        nx, ny = np.linalg.norm(xf, axis=1), np.linalg.norm(y, axis=1)
        assert np.all(np.abs(ny - nx) <= 2 ** -8 * nx)
        # inverse rotation (transpose) in float64
        h = 64
        c = t[p, :, 0].astype(np.float64); s = t[p, :, 1].astype(np.float64)
        back = np.concatenate([y[:, :h] * c + y[:, h:] * s, y[:, h:] * c - y[:, :h] * s], axis=1)
        assert np.max(np.abs(back - xf)) <= 2 ** -7 * np.max(np.abs(xf))


def test_relative_position_property():
    # <R_p q, R_p' k> depends on p - p' only (checked on unrounded rotations)
    r = np.random.Generator(np.random.PCG64(6))
    q = oracle.bf16_to_f64(bf16_normal(r, (128,)))
    k = oracle.bf16_to_f64(bf16_normal(r, (128,)))
    t = oracle.rope_table(1e6, 128, 400)
    base = None
    for shift in (0, 1, 50, 300):
        v = float(np.dot(_rot_f64(q, t, 10 + shift), _rot_f64(k, t, 3 + shift)))
        if base is None:
            base = v
        assert abs(v - base) <= 1e-5 * np.linalg.norm(q) * np.linalg.norm(k)
