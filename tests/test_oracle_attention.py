"""Pins for the oracle's paged decode attention.

Against: brute-force contiguous attention (a separate C routine and a numpy /
scipy route), closed forms (one-token context returns V, identical keys or a
zero scale return the mean of V, per-head constant V exposes the GQA head map),
paging invariance (a permutation of the physical blocks changes nothing), and
the zero row for empty contexts.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from workloads import bf16_normal

BS = 16


def _paged_from_contiguous(K, V, lens, num_blocks, r):
    """Scatter contiguous K/V [B][Hkv][n_max][d] into a paged cache through a
    random block assignment; returns caches and block tables."""
    B, Hkv, n_max, d = K.shape
    mb = -(-n_max // BS)
    perm = r.permutation(num_blocks)
    kc = np.full((num_blocks, Hkv, BS, d), 0x7FA5, np.uint16)
    vc = np.full_like(kc, 0x7FA5)
    bt = np.full((B, mb), -1, np.int32)
    nxt = 0
    for b in range(B):
        for j in range(-(-int(lens[b]) // BS)):
            blk = int(perm[nxt]); nxt += 1
            bt[b, j] = blk
            for o in range(BS):
                t = j * BS + o
                if t < lens[b]:
                    kc[blk, :, o] = K[b, :, t]
                    vc[blk, :, o] = V[b, :, t]
    return kc, vc, bt


def _case(seed, B, Hq, Hkv, d, lens, num_blocks=None):
    r = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(lens, np.int32)
    n_max = max(1, int(lens.max()))
    q = bf16_normal(r, (B, Hq, d))
    K = bf16_normal(r, (B, Hkv, n_max, d))
    V = bf16_normal(r, (B, Hkv, n_max, d))
    if num_blocks is None:
        num_blocks = int(sum(-(-int(n) // BS) for n in lens)) + 5
    kc, vc, bt = _paged_from_contiguous(K, V, lens, num_blocks, r)
    return q, K, V, kc, vc, bt, lens, r


def _numpy_attention(q, K, V, lens, scale, G):
    qf, Kf, Vf = (oracle.bf16_to_f64(a) for a in (q, K, V))
    B, Hq, d = qf.shape
    out = np.zeros((B, Hq, d))
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        for j in range(Hq):
            h = j // G
            s = scale * (Kf[b, h, :n] @ qf[b, j])
            out[b, j] = softmax(s) @ Vf[b, h, :n]
    return out


@pytest.mark.parametrize("B,Hq,Hkv,d,lens", [
    (2, 4, 2, 4, [5, 37]),
    (3, 6, 2, 64, [1, 16, 64]),
    (4, 7, 1, 4, [17, 31, 32, 33]),
    (2, 4, 4, 64, [48, 3]),
])
def test_paged_matches_contiguous_bruteforce(B, Hq, Hkv, d, lens):
    q, K, V, kc, vc, bt, lens, _ = _case(11, B, Hq, Hkv, d, lens)
    scale = 1.0 / np.sqrt(d)
    paged = oracle.paged_attention(q, kc, vc, bt, lens, scale)
    contig = oracle.contiguous_attention(q, K, V, lens, scale)
    npref = _numpy_attention(q, K, V, lens, scale, Hq // Hkv)
    assert np.max(np.abs(paged - contig)) <= 1e-12
    assert np.max(np.abs(paged - npref)) <= 1e-12


def test_paging_invariance_is_exact():
    q, K, V, kc, vc, bt, lens, r = _case(12, 3, 8, 2, 64, [40, 7, 80], num_blocks=40)
    a = oracle.paged_attention(q, kc, vc, bt, lens, 0.125)
    # move every physical block to a new random location and rewrite the tables
    perm = r.permutation(kc.shape[0])
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    b = oracle.paged_attention(q, kc2, vc2, bt2, lens, 0.125)
    assert np.array_equal(a, b)


def test_one_token_context_returns_v():
    q, K, V, kc, vc, bt, lens, _ = _case(13, 2, 4, 2, 64, [1, 1])
    out = oracle.paged_attention(q, kc, vc, bt, lens, 0.125)
    Vf = oracle.bf16_to_f64(V)
    for j in range(4):
        assert np.array_equal(out[:, j], Vf[:, j // 2, 0])


def test_identical_keys_and_zero_scale_give_mean_of_v():
    q, K, V, kc, vc, bt, lens, r = _case(14, 2, 4, 2, 64, [33, 20])
    Vf = oracle.bf16_to_f64(V)
    mean = np.stack([Vf[b, :, :lens[b]].mean(axis=1) for b in range(2)])  # [B][Hkv][d]
    out0 = oracle.paged_attention(q, kc, vc, bt, lens, 0.0)
    K1 = np.broadcast_to(K[:, :, :1], K.shape).copy()
    kc1, vc1, bt1 = _paged_from_contiguous(K1, V, lens, kc.shape[0], r)
    out1 = oracle.paged_attention(q, kc1, vc1, bt1, lens, 0.125)
    for j in range(4):
        assert np.max(np.abs(out0[:, j] - mean[:, j // 2])) <= 1e-13
        assert np.max(np.abs(out1[:, j] - mean[:, j // 2])) <= 1e-13


def test_gqa_head_map_is_repeat_interleave():
    # KV head h holds V == h + 1 everywhere, so query head j must return j // G + 1
    B, Hq, Hkv, d = 2, 12, 3, 4
    q, K, V, kc, vc, bt, lens, r = _case(15, B, Hq, Hkv, d, [9, 21])
    for h in range(Hkv):
        V[:, h] = oracle.f64_to_bf16(np.full(V[:, h].shape, float(h + 1)))
    kc, vc, bt = _paged_from_contiguous(K, V, lens, kc.shape[0], r)
    out = oracle.paged_attention(q, kc, vc, bt, lens, 0.5)
    for j in range(Hq):
        assert np.allclose(out[:, j], j // (Hq // Hkv) + 1, atol=1e-12, rtol=0)


def test_empty_context_gives_zero_row_and_large_scale_is_stable():
    q, K, V, kc, vc, bt, lens, _ = _case(16, 3, 4, 2, 64, [0, 12, 5])
    out = oracle.paged_attention(q, kc, vc, bt, lens, 1000.0)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out))
    # with a huge scale the output is the V of the best-scoring token
    Kf, Vf, qf = (oracle.bf16_to_f64(a) for a in (K, V, q))
    for b in (1, 2):
        for j in range(4):
            t = int(np.argmax(Kf[b, j // 2, :lens[b]] @ qf[b, j]))
            assert np.max(np.abs(out[b, j] - Vf[b, j // 2, t])) <= 1e-6


def test_threads_do_not_change_results():
    q, K, V, kc, vc, bt, lens, _ = _case(17, 4, 8, 2, 64, [100, 3, 47, 64])
    a = oracle.paged_attention(q, kc, vc, bt, lens, 0.125, nthreads=1)
    b = oracle.paged_attention(q, kc, vc, bt, lens, 0.125, nthreads=5)
    assert np.array_equal(a, b)
