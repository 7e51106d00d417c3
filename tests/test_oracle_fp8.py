"""Pins for the oracle's FP8 (e4m3) KV path: decoding of all 256 codes and
round-to-nearest-even encoding against torch's float8_e4m3fn (a library
routine: fp32 inputs, in range), encoding against a brute-force nearest search
over every finite code, saturation, the FP8 append as the bf16 append
followed by per-head quantisation, and FP8 attention reducing to the pinned
bf16 attention when every cached value is an e4m3 value and scales are 1,
plus exact invariance when a power of two moves between q and the K scale."""
import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_normal

BS = 16


def _torch_decode(codes):
    return torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = _torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2        # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert np.nanmax(ours) == 448.0 and ours[1] == 2.0 ** -9


def test_encode_matches_torch_on_fp32_values_in_range():
    r = np.random.Generator(np.random.PCG64(1))
    x = np.concatenate([
        r.standard_normal(20000) * 10.0,
        r.uniform(-448, 448, 20000),
        r.uniform(-2.0 ** -5, 2.0 ** -5, 20000),                       # subnormal range
        oracle.e4m3_to_f64(np.arange(0, 126, dtype=np.uint8)),            # exact codes
        (oracle.e4m3_to_f64(np.arange(0, 125, dtype=np.uint8)) +
         oracle.e4m3_to_f64(np.arange(1, 126, dtype=np.uint8))) / 2,      # midpoints: ties to even
    ]).astype(np.float32).astype(np.float64)
    ours = oracle.e4m3_from_f64(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_is_the_nearest_code_bruteforce():
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = oracle.e4m3_to_f64(finite)
    r = np.random.Generator(np.random.PCG64(2))
    x = np.concatenate([r.uniform(-460, 460, 3000), r.standard_normal(3000) * 0.01])
    got = oracle.e4m3_to_f64(oracle.e4m3_from_f64(x))
    for xi, gi in zip(x, got):
        if abs(xi) >= 448:
            assert gi == np.copysign(448.0, xi)
            continue
        dist = np.abs(vals - xi)
        best = vals[dist == dist.min()]
        if len(set(best.tolist())) > 1:                          # a tie: the even mantissa wins
            codes = finite[dist == dist.min()]
            best = vals[dist == dist.min()][(codes & 1) == 0]
        assert gi == best[0] or (gi == 0 and best[0] == 0)


def test_saturation_and_nan():
    big = np.array([448.0, 449.0, 464.0, 1e9, np.inf, -np.inf, -500.0, np.nan])
    c = oracle.e4m3_from_f64(big)
    assert c.tolist()[:7] == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert c[7] & 0x7F == 0x7F


def test_append_fp8_is_bf16_append_then_quantise():
    r = np.random.Generator(np.random.PCG64(3))
    B, Hq, Hkv, d, nb = 3, 4, 2, 64, 8
    q, k, v = (bf16_normal(r, (B, H, d)) for H in (Hq, Hkv, Hkv))
    pos = np.array([0, 17, 40], np.int32)
    slots = np.array([5, 40, 100], np.int32)
    table = oracle.rope_table(1e6, d, 64)
    ks = np.array([0.02, 0.5], np.float32)
    vs = np.array([0.01, 3.0], np.float32)
    kc16 = np.zeros((nb, Hkv, BS, d), np.uint16); vc16 = kc16.copy()
    q16, st = oracle.append(q, k, v, pos, slots, table, kc16, vc16)
    kc8 = np.zeros((nb, Hkv, BS, d), np.uint8); vc8 = kc8.copy()
    q8, st8 = oracle.append_fp8(q, k, v, pos, slots, table, ks, vs, kc8, vc8)
    assert st == st8 == 0 and np.array_equal(q16, q8)
    # the quotient is taken in IEEE single precision (numpy float32 division)
    want_k = oracle.e4m3_from_f64((oracle.bf16_to_f64(kc16).astype(np.float32) / ks[None, :, None, None])
                                  .astype(np.float64))
    want_v = oracle.e4m3_from_f64((oracle.bf16_to_f64(vc16).astype(np.float32) / vs[None, :, None, None])
                                  .astype(np.float64))
    touched = np.zeros(nb * BS, bool); touched[slots] = True
    touched = touched.reshape(nb, BS)[:, None, :, None]
    assert np.array_equal(np.where(touched, kc8, 0), np.where(touched, want_k, 0))
    assert np.array_equal(np.where(touched, vc8, 0), np.where(touched, want_v, 0))
    assert not kc8[~np.broadcast_to(touched, kc8.shape)].any()


def _fp8_case(seed, B=3, Hq=8, Hkv=2, d=64, lens=(5, 33, 70)):
    r = np.random.Generator(np.random.PCG64(seed))
    nblk = [-(-n // BS) for n in lens]
    nb = sum(nblk) + 2
    perm = r.permutation(nb)
    bt = np.full((B, max(nblk)), -1, np.int32)
    i = 0
    for b in range(B):
        for j in range(nblk[b]):
            bt[b, j] = perm[i]; i += 1
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F and abs(oracle.e4m3_to_f64(np.uint8(c))) < 8],
                      np.uint8)
    kc8 = r.choice(finite, size=(nb, Hkv, BS, d)).astype(np.uint8)
    vc8 = r.choice(finite, size=(nb, Hkv, BS, d)).astype(np.uint8)
    q = bf16_normal(r, (B, Hq, d))
    return q, kc8, vc8, bt, np.array(lens, np.int32)


def test_fp8_attention_with_unit_scales_equals_bf16_attention():
    q, kc8, vc8, bt, cl = _fp8_case(4)
    ones = np.ones(kc8.shape[1], np.float32)
    a = oracle.paged_attention_fp8(q, kc8, vc8, ones, ones, bt, cl, 0.125)
    # every e4m3 value below 8 in magnitude is a bf16 value: the same cache in bf16
    kc16 = oracle.f64_to_bf16(oracle.e4m3_to_f64(kc8))
    vc16 = oracle.f64_to_bf16(oracle.e4m3_to_f64(vc8))
    assert np.array_equal(oracle.bf16_to_f64(kc16), oracle.e4m3_to_f64(kc8))
    b = oracle.paged_attention(q, kc16, vc16, bt, cl, 0.125)
    assert np.array_equal(a, b)


def test_fp8_power_of_two_between_scale_and_q_is_exact():
    q, kc8, vc8, bt, cl = _fp8_case(5)
    ks = np.array([0.03, 0.7], np.float32)
    vs = np.array([0.2, 1.5], np.float32)
    a = oracle.paged_attention_fp8(q, kc8, vc8, ks, vs, bt, cl, 0.125)
    b = oracle.paged_attention_fp8(q, kc8, vc8, ks * 4, vs, bt, cl, 0.125 / 4)
    assert np.array_equal(a, b)
    # doubling V's scale doubles every product w * V exactly, hence the output
    c = oracle.paged_attention_fp8(q, kc8, vc8, ks, vs * 2, bt, cl, 0.125)
    assert np.array_equal(c, 2 * a)
