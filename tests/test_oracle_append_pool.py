"""Pins for the oracle's slot arithmetic, append and pool model.

Slots are checked against brute force (the flat list of every slot a table row
covers, indexed by position); append against its definition byte by byte
(rotated q and k, raw v, nothing else touched); the pool model against counting
invariants under seeded churn, all-or-nothing failure and LIFO reuse.
"""
import numpy as np
import pytest

import oracle
from oracle.pool import INVALID_ARG, OUT_OF_BLOCKS, UNKNOWN_SEQ, PoolModel
from workloads import CANARY_BF16, bf16_normal

BS = 16


def test_slot_mapping_bruteforce():
    r = np.random.Generator(np.random.PCG64(21))
    B, mb = 6, 9
    bt = np.stack([r.permutation(200)[:mb] for _ in range(B)]).astype(np.int32)
    pos = r.integers(0, mb * BS, size=B).astype(np.int32)
    got = oracle.slot_mapping(bt, pos)
    for b in range(B):
        flat = [int(blk) * BS + o for blk in bt[b] for o in range(BS)]
        assert got[b] == flat[pos[b]]


def test_append_definition():
    r = np.random.Generator(np.random.PCG64(22))
    B, Hq, Hkv, d, nb = 3, 8, 2, 64, 10
    q = bf16_normal(r, (B, Hq, d)); k = bf16_normal(r, (B, Hkv, d)); v = bf16_normal(r, (B, Hkv, d))
    kc = np.full((nb, Hkv, BS, d), CANARY_BF16, np.uint16); vc = kc.copy()
    kc0, vc0 = kc.copy(), vc.copy()
    pos = np.array([0, 17, 300], np.int32)
    slots = np.array([5 * BS + 0, 2 * BS + 1, 9 * BS + 12], np.int32)
    table = oracle.rope_table(1e6, d, 301)
    q_out, st = oracle.append(q, k, v, pos, slots, table, kc, vc)
    assert st == 0
    touched = np.zeros((nb, BS), bool)
    for b in range(B):
        assert np.array_equal(q_out[b], oracle.rope_rotate(q[b], table, int(pos[b])))
        blk, off = divmod(int(slots[b]), BS)
        touched[blk, off] = True
        assert np.array_equal(kc[blk, :, off], oracle.rope_rotate(k[b], table, int(pos[b])))
        assert np.array_equal(vc[blk, :, off], v[b])
    assert np.array_equal(kc[5, :, 0], k[0])  # position 0: unrotated
    mask = ~touched[:, None, :, None].repeat(Hkv, 1).repeat(d, 3)
    assert np.array_equal(kc[mask], kc0[mask]) and np.array_equal(vc[mask], vc0[mask])


def test_append_reports_bad_slot_and_position():
    r = np.random.Generator(np.random.PCG64(23))
    q = bf16_normal(r, (2, 2, 4)); k = bf16_normal(r, (2, 1, 4)); v = bf16_normal(r, (2, 1, 4))
    kc = np.zeros((2, 1, BS, 4), np.uint16); vc = kc.copy()
    table = oracle.rope_table(1e6, 4, 8)
    _, st = oracle.append(q, k, v, np.array([1, 2], np.int32), np.array([3, 2 * BS], np.int32), table, kc, vc)
    assert st == -1
    _, st = oracle.append(q, k, v, np.array([1, 8], np.int32), np.array([3, 4], np.int32), table, kc, vc)
    assert st == -1


def _check_invariants(p: PoolModel, num_blocks):
    owned = [blk for t in p.tables.values() for blk in t]
    assert len(owned) == len(set(owned))
    assert len(owned) + p.num_free() == num_blocks
    assert set(owned).isdisjoint(p.free_stack)
    for s, t in p.tables.items():
        assert len(t) == -(-p.tokens[s] // BS)


def test_pool_model_churn_invariants():
    r = np.random.Generator(np.random.PCG64(24))
    N = 300
    p = PoolModel(N, 40, 32, initial_order=r.permutation(N))
    for _ in range(3000):
        s = int(r.integers(0, 40))
        if r.random() < 0.3 and s in p.tables:
            assert p.free(s) == 0
        else:
            before = (list(p.free_stack), {k: list(v) for k, v in p.tables.items()})
            n = p.tokens.get(s, 0) + int(r.integers(0, 60))
            st = p.alloc(s, n)
            if st == OUT_OF_BLOCKS:
                assert (p.free_stack, p.tables) == before
            else:
                assert st in (0, INVALID_ARG)
        _check_invariants(p, N)


def test_pool_model_order_and_errors():
    p = PoolModel(8, 4, 4, initial_order=[5, 2, 7, 0, 1, 3, 4, 6])
    assert p.alloc(0, 17) == 0 and p.tables[0] == [5, 2]
    assert p.alloc(1, 16) == 0 and p.tables[1] == [7]
    assert p.alloc(0, 33) == 0 and p.tables[0] == [5, 2, 0]
    assert p.free(0) == 0
    assert p.alloc(2, 48) == 0 and p.tables[2] == [0, 2, 5]  # LIFO reuse
    assert p.free(3) == UNKNOWN_SEQ
    assert p.alloc(3, 4 * BS + 1) == INVALID_ARG  # wider than a table row
    assert p.alloc(3, 3 * BS + 1) == 0 and p.tables[3] == [1, 3, 4, 6] and p.num_free() == 0
    assert p.alloc(1, 17) == OUT_OF_BLOCKS and p.tables[1] == [7] and p.tokens[1] == 16
