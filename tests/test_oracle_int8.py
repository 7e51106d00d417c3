"""Pins for the oracle's INT8 KV path (nxmr.cn article, §2.2 "量化压缩的实战选择":
symmetric 8-bit quantisation in groups of 64 tokens, scale = 127 / max|x|,
clamp to [-128, 127], conversion to int8).

What pins it, without reusing its code:
* codes worked out by hand where 127 / m is exact (m a power of two), which
  tell truncation toward zero from rounding or flooring;
* on random groups, every code against the exact rational quotient
  |x| * 127 / m (Python fractions over the bf16 values): the code is that
  quotient truncated, except within the two single-precision roundings of an
  integer;
* exact invariance under a power-of-two rescale of the group, the zero group,
  the group's largest element at +-127 (or 126 where the roundings land just
  below 127);
* group structure by brute force: each block's stored maximum is the maximum
  over exactly its group's tokens, groups do not see each other, untouched
  bytes stay zero;
* the token-by-token append (the open group quantised again from its original
  values whenever a token joins) equals quantising the final history;
* INT8 attention reducing bit for bit to the pinned bf16 attention when every
  value is an integer and each group holds +-127 (codes = values), and exact
  doubling of the output (or of the scores) with V's (or K's) maxima."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import bf16_normal

BS = 16
GRP = 64


def _bits(vals):
    """bf16 bit patterns of float values that are bf16 numbers."""
    bits = oracle.f64_to_bf16(np.asarray(vals, np.float64))
    assert np.array_equal(oracle.bf16_to_f64(bits), np.asarray(vals, np.float64))
    return bits


def test_int8_codes_closed_forms():
    # m = 1: 127 / m = 127 exactly; x * 127 is exact in single precision
    x = [1.0, -1.0, 0.5, -0.5, 0.25, -0.25, 0.75, -0.75, 0.0, 0.125, -0.125, 2.0 ** -7, 0.99609375]
    #    127   -127  63.5 -63.5 31.75 -31.75 95.25 -95.25  0  15.875 -15.875 0.9921875 126.50390625
    want = [127, -127, 63, -63, 31, -31, 95, -95, 0, 15, -15, 0, 126]
    codes, m = oracle.int8_quantize(_bits(x))
    assert m == 1.0 and codes.tolist() == want
    # m = 4: 127 / 4 = 31.75 exactly
    x = [4.0, -4.0, 1.0, -3.0, 2.5, 0.0625]
    #    127  -127  31.75 -95.25 79.375 1.984375
    codes, m = oracle.int8_quantize(_bits(x))
    assert m == 4.0 and codes.tolist() == [127, -127, 31, -95, 79, 1]


def _exact_check(xbits, codes, m):
    """Each code against the exact quotient |x| * 127 / m."""
    xv = oracle.bf16_to_f64(xbits).ravel()
    M = Fraction(m)
    for xi, ci in zip(xv.tolist(), codes.ravel().tolist()):
        e = abs(Fraction(xi)) * 127 / M           # exact, in [0, 127]
        k = int(e)                                # truncation of the exact quotient
        c = abs(int(ci))
        assert c <= 127
        assert ci == 0 or (ci > 0) == (xi > 0)    # the sign is kept
        if c != k:
            # only where the two single-precision roundings (127 / m, then
            # x * s) move the product across an integer: within 2^-22
            # relative of one
            near = min(abs(e - k), abs(e - (k + 1)))
            assert near <= e * Fraction(1, 1 << 22), (xi, m, ci, float(e))
            assert abs(c - k) <= 1


@pytest.mark.parametrize("scale", [1.0, 1e-3, 37.0, 2.0 ** 40, 2.0 ** -40])
def test_int8_codes_against_exact_quotient(scale):
    r = np.random.Generator(np.random.PCG64(int(abs(np.log2(scale))) + 11))
    for trial in range(6):
        n = [1, 7, 64 * 128, 1000, 64 * 64, 3][trial]
        x = (r.standard_normal(n) * scale).astype(np.float32)
        if trial == 5:
            x[:] = [scale, -scale, scale]                         # ties for the maximum
        xb = oracle.f64_to_bf16(x.astype(np.float64))
        codes, m = oracle.int8_quantize(xb)
        assert m == np.abs(oracle.bf16_to_f64(xb)).max()
        _exact_check(xb, codes, m)
        top = np.abs(oracle.bf16_to_f64(xb)) == m
        assert set(np.abs(codes[top]).tolist()) <= {126, 127}


def test_int8_power_of_two_rescale_is_exact():
    r = np.random.Generator(np.random.PCG64(12))
    xb = bf16_normal(r, (GRP, 32))
    codes, m = oracle.int8_quantize(xb)
    x = oracle.bf16_to_f64(xb)
    for k in (-30, -3, 1, 9, 60):
        xs = oracle.f64_to_bf16(x * 2.0 ** k)
        assert np.array_equal(oracle.bf16_to_f64(xs), x * 2.0 ** k)
        c2, m2 = oracle.int8_quantize(xs)
        assert m2 == m * 2.0 ** k and np.array_equal(c2, codes)


def test_int8_zero_group_and_single_value():
    codes, m = oracle.int8_quantize(np.zeros(GRP * 8, np.uint16))
    assert m == 0.0 and not codes.any()
    codes, m = oracle.int8_quantize(_bits([-3.5]))
    assert m == 3.5 and codes.tolist() in ([-127], [-126])


def _history_case(seed, lens, Hkv=2, d=32, spare=3):
    r = np.random.Generator(np.random.PCG64(seed))
    B = len(lens)
    nblk = [-(-n // BS) for n in lens]
    nb = sum(nblk) + spare
    perm = r.permutation(nb)
    bt = np.full((B, max(max(nblk), 1) + 2), -1, np.int32)
    i = 0
    for b in range(B):
        for j in range(nblk[b]):
            bt[b, j] = perm[i]
            i += 1
    kc = np.zeros((nb, Hkv, BS, d), np.uint16)
    vc = np.zeros_like(kc)
    for b in range(B):
        for t in range(lens[b]):
            blk = bt[b, t // BS]
            # groups of very different ranges: group g scaled by 4^g
            kc[blk, :, t % BS] = oracle.f64_to_bf16(oracle.bf16_to_f64(bf16_normal(r, (Hkv, d))) * 4.0 ** (t // GRP))
            vc[blk, :, t % BS] = bf16_normal(r, (Hkv, d))
    slots = r.permutation(B + 2)[:B].astype(np.int32)
    return kc, vc, bt, np.array(lens, np.int32), slots, B + 2


def test_int8_history_groups_by_brute_force():
    lens = [1, 15, 16, 63, 64, 65, 130, 200]
    kc, vc, bt, cl, slots, nslot = _history_case(21, lens)
    nb, Hkv, _, d = kc.shape
    st = oracle.int8_state(nb, Hkv, d, nslot)
    assert oracle.int8_from_bf16_cache(kc, vc, bt, cl, slots, st) == 0
    touched = np.zeros((nb, BS), bool)
    for b, n in enumerate(lens):
        for src, c8, am, opn in ((kc, st["k8"], st["k_amax"], st["k_open"]), (vc, st["v8"], st["v_amax"], st["v_open"])):
            for h in range(Hkv):
                for g0 in range(0, n, GRP):
                    toks = range(g0, min(n, g0 + GRP))
                    rows = np.stack([src[bt[b, t // BS], h, t % BS] for t in toks])
                    mx = np.abs(oracle.bf16_to_f64(rows)).max()
                    for t in toks:
                        assert am[bt[b, t // BS], h] == mx                   # the group's own maximum
                    codes, m = oracle.int8_quantize(rows)
                    got = np.stack([c8[bt[b, t // BS], h, t % BS] for t in toks])
                    assert m == mx and np.array_equal(got, codes)
                    _exact_check(rows, got, mx)
                last0 = (n - 1) // GRP * GRP
                assert np.array_equal(opn[slots[b], h, : n - last0],
                                      np.stack([src[bt[b, t // BS], h, t % BS] for t in range(last0, n)]))
        for t in range(n):
            touched[bt[b, t // BS], t % BS] = True
    for c8 in (st["k8"], st["v8"]):
        assert not c8.transpose(0, 2, 1, 3)[~touched].any()               # nothing else written
    used_blocks = np.unique(np.concatenate([bt[b, : -(-n // BS)] for b, n in enumerate(lens)]))
    spare = np.setdiff1d(np.arange(nb), used_blocks)
    assert not st["k_amax"][spare].any() and not st["v_amax"][spare].any()


def test_int8_groups_do_not_see_each_other():
    lens = [150]
    kc, vc, bt, cl, slots, nslot = _history_case(22, lens)
    nb, Hkv, _, d = kc.shape
    a = oracle.int8_state(nb, Hkv, d, nslot)
    oracle.int8_from_bf16_cache(kc, vc, bt, cl, slots, a)
    # blow up one value of group 2 (tokens 128..149): groups 0 and 1 keep their codes
    kc2 = kc.copy()
    blk = bt[0, 140 // BS]
    kc2[blk, 1, 140 % BS, 3] = oracle.f64_to_bf16(np.array([1e6]))[0]
    b2 = oracle.int8_state(nb, Hkv, d, nslot)
    oracle.int8_from_bf16_cache(kc2, vc, bt, cl, slots, b2)
    for t in range(150):
        bk, off = bt[0, t // BS], t % BS
        same = np.array_equal(a["k8"][bk, 1, off], b2["k8"][bk, 1, off])
        assert same == (t < 128) or t == 140
    assert np.array_equal(a["k8"][:, 0], b2["k8"][:, 0])                    # the other head untouched


@pytest.mark.parametrize("n0", [0, 1, 50, 63, 64, 100])
def test_int8_append_token_by_token_equals_history(n0):
    r = np.random.Generator(np.random.PCG64(30 + n0))
    B, Hq, Hkv, d, steps = 3, 4, 2, 32, 70
    final = [n0 + steps, n0 + steps - 5, n0 + 1]                         # one request appends a single token
    kc, vc, bt, _, slots, nslot = _history_case(40 + n0, final, Hkv=Hkv, d=d)
    nb = kc.shape[0]
    table = oracle.rope_table(1e6, d, 512)
    # replay: bf16 append of every new token gives the bf16 history; the INT8
    # append of the same tokens must give its quantisation
    kc16 = np.zeros_like(kc); vc16 = np.zeros_like(vc)
    st = oracle.int8_state(nb, Hkv, d, nslot)
    start = [min(n0, f) for f in final]
    hist_lens = np.array(start, np.int32)
    for b in range(B):
        for t in range(start[b]):
            kc16[bt[b, t // BS], :, t % BS] = kc[bt[b, t // BS], :, t % BS]
            vc16[bt[b, t // BS], :, t % BS] = vc[bt[b, t // BS], :, t % BS]
    assert oracle.int8_from_bf16_cache(kc16, vc16, bt, hist_lens, slots, st) == 0
    lens = hist_lens.copy()
    for s in range(steps):
        grow = (lens < np.array(final)).astype(np.int32)
        newl = lens + grow
        q, k, v = (bf16_normal(r, (B, H, d)) for H in (Hq, Hkv, Hkv))
        # requests that do not grow this step: context_lens 0 appends nothing
        cl_step = np.where(grow > 0, newl, 0).astype(np.int32)
        q8, s8 = oracle.append_int8(q, k, v, table, bt, cl_step, slots, st)
        pos = np.maximum(cl_step - 1, 0)
        sm = np.where(grow > 0, oracle.slot_mapping(bt, pos), -1).astype(np.int32)
        q16, s16 = oracle.append(q, k, v, pos, sm, table, kc16, vc16)
        assert s8 == 0
        assert np.array_equal(q8[grow > 0], q16[grow > 0])
        lens = newl
    want = oracle.int8_state(nb, Hkv, d, nslot)
    assert oracle.int8_from_bf16_cache(kc16, vc16, bt, lens, slots, want) == 0
    for key in ("k8", "v8", "k_amax", "v_amax"):
        assert np.array_equal(st[key], want[key]), key
    for b in range(B):                                                     # the open group's live rows
        o = (lens[b] - 1) % GRP + 1
        assert np.array_equal(st["k_open"][slots[b], :, :o], want["k_open"][slots[b], :, :o])
        assert np.array_equal(st["v_open"][slots[b], :, :o], want["v_open"][slots[b], :, :o])


def test_int8_append_rejects_bad_slot_and_block():
    B, Hq, Hkv, d = 2, 2, 1, 16
    r = np.random.Generator(np.random.PCG64(5))
    q, k, v = (bf16_normal(r, (B, H, d)) for H in (Hq, Hkv, Hkv))
    table = oracle.rope_table(1e6, d, 64)
    bt = np.array([[0, 1], [7, -1]], np.int32)
    st = oracle.int8_state(4, Hkv, d, 2)
    _, s = oracle.append_int8(q, k, v, table, bt, np.array([3, 1], np.int32), np.array([0, 1], np.int32), st)
    assert s == -1                                                          # block 7 out of range
    assert st["k8"][0, 0, 2].any() and not st["k8"][3].any()
    st = oracle.int8_state(4, Hkv, d, 2)
    _, s = oracle.append_int8(q, k, v, table, bt, np.array([3, 0], np.int32), np.array([5, 0], np.int32), st)
    assert s == -1 and not st["k8"].any()                                   # slot 5 out of range


def _int8_attn_case(seed, B=3, Hq=8, Hkv=2, d=64, lens=(5, 70, 140)):
    r = np.random.Generator(np.random.PCG64(seed))
    nblk = [-(-n // BS) for n in lens]
    nb = sum(nblk) + 2
    perm = r.permutation(nb)
    bt = np.full((B, max(nblk)), -1, np.int32)
    i = 0
    for b in range(B):
        for j in range(nblk[b]):
            bt[b, j] = perm[i]
            i += 1
    k8 = r.integers(-127, 128, size=(nb, Hkv, BS, 64 if d == 64 else d)).astype(np.int8)
    v8 = r.integers(-127, 128, size=k8.shape).astype(np.int8)
    q = bf16_normal(r, (B, Hq, d))
    return q, k8, v8, bt, np.array(lens, np.int32)


def test_int8_attention_integer_values_equal_bf16_attention():
    q, k8, v8, bt, cl = _int8_attn_case(6)
    amax = np.full(k8.shape[:2], 127.0, np.float32)                          # codes = values
    a = oracle.paged_attention_int8(q, k8, v8, amax, amax, bt, cl, 0.01)
    kc16 = oracle.f64_to_bf16(k8.astype(np.float64))                         # integers below 128: exact in bf16
    vc16 = oracle.f64_to_bf16(v8.astype(np.float64))
    b = oracle.paged_attention(q, kc16, vc16, bt, cl, 0.01)
    assert np.array_equal(a, b)


def test_int8_attention_scaling_by_two_is_exact():
    q, k8, v8, bt, cl = _int8_attn_case(7)
    r = np.random.Generator(np.random.PCG64(8))
    ka = oracle.bf16_to_f64(oracle.f64_to_bf16(r.uniform(0.5, 4.0, k8.shape[:2]))).astype(np.float32)
    va = oracle.bf16_to_f64(oracle.f64_to_bf16(r.uniform(0.5, 4.0, k8.shape[:2]))).astype(np.float32)
    a = oracle.paged_attention_int8(q, k8, v8, ka, va, bt, cl, 0.02)
    assert np.array_equal(oracle.paged_attention_int8(q, k8, v8, ka, va * 2, bt, cl, 0.02), 2 * a)
    assert np.array_equal(oracle.paged_attention_int8(q, k8, v8, ka * 2, va, bt, cl, 0.02),
                          oracle.paged_attention_int8(q, k8, v8, ka, va, bt, cl, 0.04))
    # a block's own maximum weighs only its own tokens: zeroing one block's V
    # maximum equals zeroing its codes
    blk = bt[2, 3]
    va0 = va.copy(); va0[blk] = 0
    v0 = v8.copy(); v0[blk] = 0
    assert np.array_equal(oracle.paged_attention_int8(q, k8, v8, ka, va0, bt, cl, 0.02),
                          oracle.paged_attention_int8(q, k8, v0, ka, va, bt, cl, 0.02))


def test_int8_append_tokens_equals_history():
    """Many new tokens per request through the oracle's chunked helper (the
    token-by-token append in order) give the quantisation of the final
    history, from every phase of a group, with chunks crossing groups."""
    r = np.random.Generator(np.random.PCG64(90))
    Hq, Hkv, d = 4, 2, 32
    hist = [0, 1, 63, 64, 100, 10]
    m = [70, 1, 2, 129, 28, 0]
    final = [h + c for h, c in zip(hist, m)]
    kc, vc, bt, _, slots, nslot = _history_case(91, [max(f, 1) for f in final], Hkv=Hkv, d=d)
    nb = kc.shape[0]
    table = oracle.rope_table(1e6, d, 512)
    kc16, vc16 = np.zeros_like(kc), np.zeros_like(vc)
    for b in range(len(hist)):
        for t in range(hist[b]):
            kc16[bt[b, t // BS], :, t % BS] = kc[bt[b, t // BS], :, t % BS]
            vc16[bt[b, t // BS], :, t % BS] = vc[bt[b, t // BS], :, t % BS]
    st = oracle.int8_state(nb, Hkv, d, nslot)
    assert oracle.int8_from_bf16_cache(kc16, vc16, bt, np.array(hist, np.int32), slots, st) == 0
    qs = np.concatenate([[0], np.cumsum(m)]).astype(np.int32)
    T = int(qs[-1])
    q, k, v = (bf16_normal(r, (T, H, d)) for H in (Hq, Hkv, Hkv))
    q_out, s = oracle.append_int8_tokens(q, k, v, table, bt, np.array(final, np.int32), qs, slots, st)
    assert s == 0
    # the bf16 history the same tokens make, one bf16 append per token
    for b in range(len(hist)):
        for i in range(m[b]):
            p = hist[b] + i
            row = qs[b] + i
            qo, s16 = oracle.append(q[row:row + 1], k[row:row + 1], v[row:row + 1], np.array([p], np.int32),
                                    oracle.slot_mapping(bt[b:b + 1], np.array([p], np.int32)), table, kc16, vc16)
            assert s16 == 0 and np.array_equal(qo[0], q_out[row])
    want = oracle.int8_state(nb, Hkv, d, nslot)
    assert oracle.int8_from_bf16_cache(kc16, vc16, bt, np.array(final, np.int32), slots, want) == 0
    for key in ("k8", "v8", "k_amax", "v_amax"):
        assert np.array_equal(st[key], want[key]), key
    for b in range(len(hist)):
        if final[b] > 0:
            o = (final[b] - 1) % GRP + 1
            assert np.array_equal(st["k_open"][slots[b], :, :o], want["k_open"][slots[b], :, :o])
