"""Pins for the oracle's swap model: block copies reduce to numpy fancy
indexing when destinations are distinct; a swap-out / scribble / swap-in round
trip leaves the decode attention of the swapped sequence unchanged bit for bit
(checked with the attention oracle over the old and the new table); the
LIFO free list hands an immediately swapped-in sequence its own blocks in
reverse order; a swap-in that does not fit changes nothing; and the LRU
victim equals a brute-force scan of an independent log of uses."""
import numpy as np

import oracle
from oracle.pool import INVALID_ARG, OK, OUT_OF_BLOCKS, UNKNOWN_SEQ, PoolModel
from oracle.swap import copy_blocks
from workloads import bf16_normal

BS = 16


def test_copy_reduces_to_fancy_indexing():
    r = np.random.Generator(np.random.PCG64(1))
    src = r.integers(0, 1 << 16, size=(20, 2, BS, 8), dtype=np.uint16)
    dst = r.integers(0, 1 << 16, size=(12, 2, BS, 8), dtype=np.uint16)
    si = r.choice(20, size=7, replace=True)
    di = r.choice(12, size=7, replace=False)
    want = dst.copy()
    want[di] = src[si]
    copy_blocks(src, si, dst, di)
    assert np.array_equal(dst, want)


def test_round_trip_keeps_attention_bitwise():
    r = np.random.Generator(np.random.PCG64(2))
    nb, Hkv, Hq, d = 32, 2, 4, 64
    dev = PoolModel(nb, 8, 8, r.permutation(nb))
    host = PoolModel(16, 8, 8)
    kc = bf16_normal(r, (nb, Hkv, BS, d))
    vc = bf16_normal(r, (nb, Hkv, BS, d))
    hk = np.zeros((16, Hkv, BS, d), np.uint16)
    hv = np.zeros_like(hk)
    assert dev.alloc(0, 70) == OK and dev.alloc(1, 33) == OK
    q = bf16_normal(r, (1, Hq, d))
    bt0, cl0, _ = dev.batch_meta([1])
    before = oracle.paged_attention(q, kc, vc, bt0, cl0, 0.125)
    st, table = dev.swap_out(1)
    assert st == OK and table == list(bt0[0, :3])
    assert host.alloc(1, dev.tokens[1]) == OK
    copy_blocks(kc, table, hk, host.tables[1])
    copy_blocks(vc, table, hv, host.tables[1])
    # another sequence takes the freed blocks and overwrites them
    assert dev.alloc(2, 3 * BS) == OK
    for blk in dev.tables[2]:
        kc[blk] = 0x7FA5
        vc[blk] = 0x7FA5
    st, new = dev.swap_in(1)
    assert st == OK and len(new) == 3 and not set(new) & set(dev.tables[2])
    copy_blocks(hk, host.tables[1], kc, new)
    copy_blocks(hv, host.tables[1], vc, new)
    assert host.free(1) == OK
    bt1, cl1, _ = dev.batch_meta([1])
    assert list(bt1[0, :3]) == new and cl1[0] == 33
    after = oracle.paged_attention(q, kc, vc, bt1, cl1, 0.125)
    assert np.array_equal(before, after)


def test_immediate_swap_in_returns_own_blocks_reversed_and_counts():
    p = PoolModel(40, 4, 8, np.random.Generator(np.random.PCG64(3)).permutation(40))
    assert p.alloc(0, 100) == OK
    free0 = p.num_free()
    st, t = p.swap_out(0)
    assert st == OK and p.num_free() == free0 + 7
    assert p.alloc(0, 120) == INVALID_ARG            # not resident
    assert p.swap_out(0)[0] == UNKNOWN_SEQ
    st, t2 = p.swap_in(0)
    assert st == OK and t2 == t[::-1] and p.num_free() == free0
    assert p.tokens[0] == 100


def test_swap_in_that_does_not_fit_changes_nothing():
    p = PoolModel(10, 4, 10)
    assert p.alloc(0, 64) == OK
    assert p.swap_out(0)[0] == OK
    assert p.alloc(1, 10 * BS - 16) == OK             # 9 blocks: one left
    stack = list(p.free_stack)
    assert p.swap_in(0) == (OUT_OF_BLOCKS, [])
    assert p.free_stack == stack and 0 in p.swapped and 0 not in p.tables
    assert p.free(0) == OK and 0 not in p.tokens      # a swapped sequence can be dropped


def test_lru_victim_matches_bruteforce_log():
    r = np.random.Generator(np.random.PCG64(4))
    p = PoolModel(400, 12, 16)
    log = []  # independent record: (tick, seq) of every use
    tick = 0
    for _ in range(400):
        op = int(r.integers(0, 5))
        s = int(r.integers(0, 12))
        if op == 0:
            n = p.tokens.get(s, 0) + int(r.integers(1, 40))
            if p.alloc(s, n) == OK:
                tick += 1
                log.append((tick, s))
        elif op == 1 and s in p.tables:
            seqs = sorted({s, int(r.integers(0, 12))} & set(p.tables))
            assert p.touch(seqs) == OK
            tick += 1
            log.extend((tick, x) for x in seqs)
        elif op == 2:
            p.swap_out(s)
        elif op == 3 and s in p.swapped:
            if p.swap_in(s)[0] == OK:
                tick += 1
                log.append((tick, s))
        elif op == 4 and r.random() < 0.2:
            p.free(s)
        excl = [int(x) for x in r.choice(12, size=int(r.integers(0, 3)), replace=False)]
        # brute force: last use of each resident, block-holding sequence since it became resident
        best = None
        for cand in range(12):
            if cand not in p.tables or not p.tables[cand] or cand in excl:
                continue
            last = max([t for t, x in log if x == cand], default=0)
            if best is None or (last, cand) < best:
                best = (last, cand)
        assert p.lru_victim(excl) == (best[1] if best else -1)
