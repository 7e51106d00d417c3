"""Swap-out / swap-in and LRU bookkeeping of the library pool against the
oracle's pool model: the same random sequence of alloc, touch, swap, free and
victim queries gives the same statuses, tables, free counts and victims."""
import numpy as np
import pytest

from oracle.pool import PoolModel


@pytest.fixture(scope="module")
def mi():
    import paged_kv_decode_25_gb300 as m
    from paged_kv_decode_25_gb300 import build
    build.build()
    return m


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_swap_ops_match_model(mi, seed):
    r = np.random.Generator(np.random.PCG64(seed))
    nb, ns, mb = 300, 16, 24
    order = r.permutation(nb).astype(np.int32)
    lib, model = mi.Pool(nb, ns, mb, order), PoolModel(nb, ns, mb, order)
    for _ in range(1500):
        op = int(r.integers(0, 6))
        s = int(r.integers(0, ns))
        if op == 0:
            n = int(model.tokens.get(s, 0)) + int(r.integers(0, 60))
            assert lib.alloc(s, n) == model.alloc(s, n)
        elif op == 1:
            assert lib.swap_out(s) == model.swap_out(s)
        elif op == 2:
            assert lib.swap_in(s) == model.swap_in(s)
        elif op == 3:
            seqs = sorted(set(int(x) for x in r.integers(0, ns, size=int(r.integers(1, 4)))))
            assert lib.touch(seqs) == model.touch(seqs)
        elif op == 4 and r.random() < 0.3:
            assert lib.free(s) == model.free(s)
        excl = [int(x) for x in r.choice(ns, size=int(r.integers(0, 4)), replace=False)]
        assert lib.lru_victim(excl) == model.lru_victim(excl)
        assert lib.num_free() == model.num_free()
    resident = sorted(model.tables)
    if resident:
        bt, cl, _ = lib.batch_meta(resident)
        bt_m, cl_m, _ = model.batch_meta(resident)
        assert np.array_equal(bt, bt_m) and np.array_equal(cl, cl_m)


def test_swapped_sequences_are_not_resident(mi):
    p = mi.Pool(20, 4, 8)
    assert p.alloc(0, 40) == 0 and p.alloc(1, 17) == 0
    st, blocks = p.swap_out(0)
    assert st == 0 and len(blocks) == 3 and p.num_free() == 20 - 2
    st, _, _, _ = mi.mi_kv_pool_batch_meta(p.handle, [0], 8)
    assert st == mi.MI_ERR_UNKNOWN_SEQ
    assert mi.mi_kv_pool_token_slots(p.handle, 0, 0, 1)[0] == mi.MI_ERR_UNKNOWN_SEQ
    assert mi.mi_kv_pool_seq_blocks(p.handle, 0) is None
    assert p.alloc(0, 50) == mi.MI_ERR_INVALID_ARG
    assert p.touch([0]) == mi.MI_ERR_UNKNOWN_SEQ
    assert p.lru_victim() == 1
    st, new = p.swap_in(0)
    assert st == 0 and new == blocks[::-1]
    assert mi.mi_kv_pool_swap_out(p.handle, 0, max_out=2)[0] == mi.MI_ERR_INVALID_ARG  # 3 blocks held
    assert mi.mi_kv_pool_swap_in(p.handle, 0)[0] == mi.MI_ERR_UNKNOWN_SEQ              # resident
