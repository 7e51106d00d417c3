"""Pins for the oracle's causal paged prefill attention and token slots.

Against: the decode oracle (one new token per request is exactly decode),
brute-force causal softmax attention over contiguous K/V (numpy + scipy),
causality (perturbing keys after a token's position leaves that token's output
unchanged), the position-0 closed form (a request's very first token returns
its own V), and a brute-force slot list for the pool model's token slots.
"""
import numpy as np
from scipy.special import softmax

import oracle
from oracle.pool import PoolModel
from workloads import bf16_normal

BS = 16


def _case(seed, Hq, Hkv, d, lens, news):
    """Paged caches holding each request's full context (history + new
    tokens), block tables, and q rows for the new tokens."""
    r = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(lens, np.int32)
    news = np.asarray(news, np.int32)
    R = len(lens)
    n_max = int(lens.max())
    K = bf16_normal(r, (R, Hkv, n_max, d))
    V = bf16_normal(r, (R, Hkv, n_max, d))
    nblk = [-(-int(n) // BS) for n in lens]
    nb = sum(nblk) + 3
    perm = r.permutation(nb)
    bt = np.full((R, max(nblk)), -1, np.int32)
    kc = np.full((nb, Hkv, BS, d), 0x7FA5, np.uint16)
    vc = kc.copy()
    i = 0
    for b in range(R):
        for j in range(nblk[b]):
            blk = int(perm[i]); i += 1
            bt[b, j] = blk
            m = min(BS, int(lens[b]) - j * BS)
            kc[blk, :, :m] = K[b, :, j * BS: j * BS + m]
            vc[blk, :, :m] = V[b, :, j * BS: j * BS + m]
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    q = bf16_normal(r, (int(qs[-1]), Hq, d))
    return q, K, V, kc, vc, bt, lens, qs


def test_one_new_token_is_decode():
    q, K, V, kc, vc, bt, lens, qs = _case(1, 8, 2, 64, [5, 40, 16, 33], [1, 1, 1, 1])
    a = oracle.paged_prefill_attention(q, kc, vc, bt, lens, qs, 0.125)
    b = oracle.paged_attention(q, kc, vc, bt, lens, 0.125)
    assert np.array_equal(a, b)


def test_matches_bruteforce_causal_softmax():
    Hq, Hkv, d = 6, 2, 64
    lens, news = [40, 17, 64, 3], [7, 17, 33, 1]
    q, K, V, kc, vc, bt, lens, qs = _case(2, Hq, Hkv, d, lens, news)
    out = oracle.paged_prefill_attention(q, kc, vc, bt, lens, qs, 0.125, nthreads=3)
    qf, Kf, Vf = (oracle.bf16_to_f64(x) for x in (q, K, V))
    G = Hq // Hkv
    for r in range(len(lens)):
        m, n = int(qs[r + 1] - qs[r]), int(lens[r])
        for i in range(m):
            pos = n - m + i
            for j in range(Hq):
                s = 0.125 * (Kf[r, j // G, : pos + 1] @ qf[qs[r] + i, j])
                ref = softmax(s) @ Vf[r, j // G, : pos + 1]
                assert np.max(np.abs(out[qs[r] + i, j] - ref)) <= 1e-12


def test_future_keys_do_not_matter():
    q, K, V, kc, vc, bt, lens, qs = _case(3, 4, 1, 64, [48], [20])
    a = oracle.paged_prefill_attention(q, kc, vc, bt, lens, qs, 0.125)
    # scramble keys and values of the last 12 positions (28 .. 47)
    kc2, vc2 = kc.copy(), vc.copy()
    for t in range(36, 48):
        blk = bt[0, t // BS]
        kc2[blk, :, t % BS] = 0x3F80
        vc2[blk, :, t % BS] = 0xC000
    b = oracle.paged_prefill_attention(q, kc2, vc2, bt, lens, qs, 0.125)
    first_changed = 36 - (48 - 20)  # new-token index of position 36
    assert np.array_equal(a[:first_changed], b[:first_changed])
    assert not np.array_equal(a[first_changed:], b[first_changed:])


def test_first_token_returns_its_own_v():
    q, K, V, kc, vc, bt, lens, qs = _case(4, 4, 2, 64, [9, 20], [9, 20])  # no history: positions start at 0
    out = oracle.paged_prefill_attention(q, kc, vc, bt, lens, qs, 0.3)
    Vf = oracle.bf16_to_f64(V)
    for r in range(2):
        for j in range(4):
            assert np.array_equal(out[qs[r], j], Vf[r, j // 2, 0])


def test_pool_model_token_slots_bruteforce():
    p = PoolModel(40, 3, 8, initial_order=np.random.Generator(np.random.PCG64(5)).permutation(40))
    assert p.alloc(0, 50) == 0 and p.alloc(1, 17) == 0 and p.alloc(0, 90) == 0
    flat = [blk * BS + o for blk in p.tables[0] for o in range(BS)]
    assert list(p.token_slots(0, 45, 30)) == flat[45:75]
