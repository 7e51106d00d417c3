"""CPU tests of the C ABI: the library loads and exports every symbol the
header declares; the host block pool matches the oracle's pool model table for
table under each workload's history and random churn; host-side argument checks
reject bad calls without touching a GPU; the host RoPE table matches the
oracle's bit for bit."""
import os
import re

import numpy as np
import pytest

import oracle
from oracle.pool import PoolModel
from workloads import WORKLOADS, context_lengths, initial_free_order, setup_pool

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mi():
    import paged_kv_decode_25_gb300 as mi
    from paged_kv_decode_25_gb300 import build
    build.build()
    mi.load()
    return mi


def _declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mi_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(mi):
    declared = _declared_symbols()
    assert declared, "no declarations found"
    lib = mi.load()
    for n in declared:
        assert hasattr(lib, n), n
    assert declared == set(mi.EXPORTS)


def test_header_constants_match_the_binding(mi):
    """Every numeric #define of the header has the binding's value."""
    src = open(os.path.join(ROOT, "include", "mi.h")).read()
    found = 0
    for name, val in re.findall(r"^#define (MI_\w+)\s+\(?([0-9xXa-fA-F]+)u?", src, flags=re.M):
        if name == "MI_NOALLOC_SCRATCH_BYTES":
            continue  # a product, checked below
        assert getattr(mi, name) == int(val, 0), name
        found += 1
    assert found >= 14
    assert mi.MI_NOALLOC_SCRATCH_BYTES == 16 * 1024 * 1024


def _compare(lib, model, seqs, mbps):
    bt1, cl1, sl1 = lib.batch_meta(seqs)
    bt2, cl2, sl2 = model.batch_meta(seqs)
    assert np.array_equal(bt1, bt2) and np.array_equal(cl1, cl2) and np.array_equal(sl1, sl2)
    assert lib.num_free() == model.num_free()
    return bt1, cl1, sl1


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_pool_matches_model_on_workload_history(mi, name):
    w = WORKLOADS[name]
    ctx = context_lengths(w)
    order = initial_free_order(w)
    lib = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    model = PoolModel(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    setup_pool(w, lib, ctx)
    setup_pool(w, model, ctx)
    seqs = list(range(w.B))
    _compare(lib, model, seqs, w.max_blocks_per_seq)
    steps = min(w.sweep_steps, 20)
    for s in range(steps):
        for b in seqs:
            assert lib.alloc(b, int(ctx[b]) + s + 1) == 0
            assert model.alloc(b, int(ctx[b]) + s + 1) == 0
        bt, cl, sl = _compare(lib, model, seqs, w.max_blocks_per_seq)
        # the slot of the newest token, from the oracle's own slot arithmetic
        assert np.array_equal(sl, oracle.slot_mapping(bt, cl - 1))
    if w.churn:  # the churned pool hands out blocks out of order
        bt, _, _ = lib.batch_meta(seqs)
        assert np.any(np.diff(bt[0][bt[0] >= 0]) != 1)


def test_pool_random_churn_matches_model(mi):
    r = np.random.Generator(np.random.PCG64(31))
    N, S, W = 500, 64, 40
    order = r.permutation(N)
    lib = mi.Pool(N, S, W, order)
    model = PoolModel(N, S, W, order)
    for it in range(4000):
        s = int(r.integers(0, S))
        if r.random() < 0.25:
            assert lib.free(s) == model.free(s)
        else:
            n = max(0, model.tokens.get(s, 0) + int(r.integers(-3, 80)))
            assert lib.alloc(s, n) == model.alloc(s, n)
        if it % 97 == 0:
            live = sorted(model.tables)
            if live:
                _compare(lib, model, live, W)
    for s in sorted(model.tables):
        got = mi.mi_kv_pool_seq_blocks(lib.handle, s)
        assert list(got) == model.tables[s]


def test_pool_errors(mi):
    st, h = mi.mi_kv_pool_create(8, 16, 2, 2)
    assert st == mi.MI_OK
    assert mi.mi_kv_pool_alloc(h, 2, 1) == mi.MI_ERR_INVALID_ARG      # seq id out of range
    assert mi.mi_kv_pool_alloc(h, 0, -1) == mi.MI_ERR_INVALID_ARG     # negative tokens
    assert mi.mi_kv_pool_alloc(h, 0, 33) == mi.MI_ERR_INVALID_ARG     # wider than a row
    assert mi.mi_kv_pool_free(h, 1) == mi.MI_ERR_UNKNOWN_SEQ
    assert mi.mi_kv_pool_alloc(h, 0, 20) == mi.MI_OK
    assert mi.mi_kv_pool_alloc(h, 0, 10) == mi.MI_ERR_INVALID_ARG     # shrinking
    st, bt, cl, sl = mi.mi_kv_pool_batch_meta(h, [0, 1], 2)
    assert st == mi.MI_ERR_UNKNOWN_SEQ
    mi.mi_kv_pool_destroy(h)
    assert mi.mi_kv_pool_create(8, 32, 2, 2)[0] == mi.MI_ERR_UNSUPPORTED
    assert mi.mi_kv_pool_create(0, 16, 2, 2)[0] == mi.MI_ERR_INVALID_ARG
    assert mi.mi_kv_pool_create(4, 16, 2, 2, [0, 1, 1, 3])[0] == mi.MI_ERR_INVALID_ARG
    assert mi.mi_kv_pool_num_free(None) == -1


def test_pool_exhaustion_is_all_or_nothing(mi):
    lib = mi.Pool(6, 4, 8)
    assert lib.alloc(0, 16 * 4) == 0
    before = mi.mi_kv_pool_seq_blocks(lib.handle, 0).tolist(), lib.num_free()
    assert lib.alloc(0, 16 * 7) == mi.MI_ERR_OUT_OF_BLOCKS
    assert (mi.mi_kv_pool_seq_blocks(lib.handle, 0).tolist(), lib.num_free()) == before
    assert lib.alloc(1, 16 * 3) == mi.MI_ERR_OUT_OF_BLOCKS
    assert mi.mi_kv_pool_seq_blocks(lib.handle, 1) is None


def _state(mi, lib, S):
    """Every sequence's table, the free count and the LRU order (victims
    taken one after another)."""
    tables = [None if (t := mi.mi_kv_pool_seq_blocks(lib.handle, s)) is None else t.tolist() for s in range(S)]
    order, ex = [], []
    while (v := mi.mi_kv_pool_lru_victim(lib.handle, ex)) >= 0:
        order.append(v)
        ex.append(v)
    return tables, lib.num_free(), order


def test_pool_alloc_batch_equals_sequential_allocs(mi):
    """A batch grows its sequences exactly as the same allocs one by one:
    tables, free count and use order, repeated ids included (the pool is
    large enough that every batch fits)."""
    r = np.random.Generator(np.random.PCG64(41))
    S, W = 24, 32
    N = S * W
    order = r.permutation(N)
    a, b = mi.Pool(N, S, W, order), mi.Pool(N, S, W, order)
    tok = np.zeros(S, np.int64)
    for it in range(300):
        if r.random() < 0.2:
            s = int(r.integers(0, S))
            assert a.free(s) == b.free(s)
            tok[s] = 0
            continue
        k = int(r.integers(1, 9))
        seqs = r.integers(0, S, size=k)
        ntok = []
        for s in seqs:  # growing; repeated ids grow again
            tok[s] = min(int(tok[s]) + int(r.integers(0, 40)), W * 16)
            ntok.append(int(tok[s]))
        assert a.alloc_batch(seqs, ntok) == mi.MI_OK
        assert all(b.alloc(int(s), n) == mi.MI_OK for s, n in zip(seqs, ntok))
        assert _state(mi, a, S) == _state(mi, b, S)


def test_pool_alloc_batch_is_all_or_nothing(mi):
    lib = mi.Pool(10, 4, 8)
    assert lib.alloc_batch([0, 1], [16, 16]) == mi.MI_OK
    before = _state(mi, lib, 4)
    # more blocks than are free: nothing changes
    assert lib.alloc_batch([2, 3, 0], [16 * 3, 16 * 3, 16 * 4]) == mi.MI_ERR_OUT_OF_BLOCKS  # 9 of 8 free
    assert _state(mi, lib, 4) == before
    # a bad entry after good ones: nothing changes
    for seqs, ntok in (([2, 0], [16, 8]),        # shrinking sequence 0
                       ([2, 4], [16, 16]),       # id out of range
                       ([2, 3], [16, -1]),       # negative count
                       ([2, 3], [16, 16 * 9]),   # wider than a table row
                       ([2, 2], [32, 16])):      # shrinking within the batch
        assert lib.alloc_batch(seqs, ntok) == mi.MI_ERR_INVALID_ARG
        assert _state(mi, lib, 4) == before
    assert lib.alloc_batch([], []) == mi.MI_OK
    assert lib.alloc_batch([2, 2], [16, 48]) == mi.MI_OK
    assert mi.mi_kv_pool_seq_blocks(lib.handle, 2).size == 3


@pytest.mark.parametrize("d,theta,max_pos", [(64, 1e6, 100), (128, 1e6, 9000), (128, 1e4, 33)])
def test_rope_table_matches_oracle_bits(mi, d, theta, max_pos):
    st, t = mi.mi_rope_table(theta, d, max_pos)
    assert st == mi.MI_OK
    ref = oracle.rope_table(theta, d, max_pos)
    assert np.array_equal(t.view(np.uint32), ref.view(np.uint32))


def test_device_entry_points_reject_bad_args_without_a_gpu(mi):
    d = mi.dims(2, 4, 2, 64, 8, 4)
    bad = mi.dims(2, 4, 3, 64, 8, 4)  # Hq % Hkv != 0
    assert mi.mi_paged_decode_workspace_bytes(bad) == 0
    assert mi.mi_paged_kv_append(bad, 16, 16, 16, 16, 16, 16, 4, 16, 16, 16, stream=0) == mi.MI_ERR_UNSUPPORTED
    odd = mi.dims(2, 4, 2, 96, 8, 4)
    assert mi.mi_paged_kv_append(odd, 16, 16, 16, 16, 16, 16, 4, 16, 16, 16, stream=0) == mi.MI_ERR_UNSUPPORTED
    wide = mi.dims(2, 18, 2, 64, 8, 4)  # G = 9
    assert mi.load().mi_paged_decode_attention_variant(
        __import__("ctypes").byref(wide), 16, 16, 16, 16, 16, 1.0, 16, 16, 1 << 20, None, 0, 0, 0
    ) == mi.MI_ERR_UNSUPPORTED
    # null pointers are caught before any CUDA call
    assert mi.mi_paged_kv_append(d, None, 16, 16, 16, 16, 16, 4, 16, 16, 16, stream=0) == mi.MI_ERR_INVALID_ARG
    assert mi.mi_paged_decode_attention(d, None, 16, 16, 16, 16, 1.0, 16, 16, workspace_bytes=1 << 20,
                                        stream=0) == mi.MI_ERR_INVALID_ARG
    # misaligned caches are rejected
    assert mi.mi_paged_decode_attention(d, 16, 18, 16, 16, 16, 1.0, 16, 16, workspace_bytes=1 << 20,
                                        stream=0) == mi.MI_ERR_INVALID_ARG
    # an empty batch is a no-op
    zero = mi.dims(0, 4, 2, 64, 8, 4)
    assert mi.mi_paged_kv_append(zero, None, None, None, None, None, None, 4, None, None, None,
                                 stream=0) == mi.MI_OK


def test_step_rejects_bad_args_without_a_gpu(mi):
    """mi_paged_decode_step refuses bad arguments before any CUDA call: the
    addresses below are never dereferenced."""
    d = mi.dims(2, 4, 2, 64, 8, 4)
    a = {n: (i + 1) << 20 for i, n in enumerate(("q", "k", "v", "rope", "bt", "cl", "qo", "kc", "vc", "out", "ws"))}

    def step(dims=d, max_pos=64, **over):
        x = dict(a, **over)
        return mi.mi_paged_decode_step(dims, x["q"], x["k"], x["v"], x["rope"], max_pos, x["bt"], x["cl"], 0.125,
                                       x["qo"], x["kc"], x["vc"], x["out"], x["ws"], workspace_bytes=1 << 20,
                                       stream=0)
    assert step(dims=mi.dims(2, 4, 3, 64, 8, 4)) == mi.MI_ERR_UNSUPPORTED  # Hq % Hkv != 0
    for name in ("q", "k", "v", "rope", "bt", "cl", "qo", "kc", "vc", "out", "ws"):
        assert step(**{name: None}) == mi.MI_ERR_INVALID_ARG, name
    for name in ("q", "k", "v", "rope", "qo", "kc", "vc", "out", "ws"):
        assert step(**{name: a[name] + 8}) == mi.MI_ERR_INVALID_ARG, name  # not 16-byte aligned
    assert step(max_pos=0) == mi.MI_ERR_INVALID_ARG
    # q and q_out overlap (any shared byte of the B x Hq x d bf16 rows)
    assert step(qo=a["q"] + 16) == mi.MI_ERR_INVALID_ARG
    assert step(qo=a["q"] - 2 * 4 * 64 * 2 + 16) == mi.MI_ERR_INVALID_ARG
    # an empty batch is a no-op
    assert step(dims=mi.dims(0, 4, 2, 64, 8, 4)) == mi.MI_OK
    # flags: only MI_STEP_EARLY_START is defined
    for bad in (2, 0x80000000, mi.MI_STEP_EARLY_START | 4):
        assert mi.mi_paged_decode_step(d, a["q"], a["k"], a["v"], a["rope"], 64, a["bt"], a["cl"], 0.125, a["qo"],
                                       a["kc"], a["vc"], a["out"], a["ws"], workspace_bytes=1 << 20, stream=0,
                                       flags=bad) == mi.MI_ERR_INVALID_ARG
        assert mi.mi_paged_decode_step_fp8(d, a["q"], a["k"], a["v"], a["rope"], 64, a["bt"], a["cl"], a["k"],
                                           a["v"], 0.125, a["qo"], a["kc"], a["vc"], a["out"], a["ws"],
                                           workspace_bytes=1 << 20, stream=0, flags=bad) == mi.MI_ERR_INVALID_ARG
    assert step(dims=mi.dims(0, 4, 2, 64, 8, 4)) == mi.MI_OK


def test_fp8_entry_points_reject_bad_args_without_a_gpu(mi):
    """The e4m3 append and attention refuse missing scales, misaligned
    buffers and unsupported shapes before any CUDA call."""
    d = mi.dims(2, 4, 2, 64, 8, 4)
    A = 1 << 20

    def app(dims=d, ks=9 * A, vs=10 * A, kc=7 * A):
        return mi.mi_paged_kv_append_fp8(dims, A, 2 * A, 3 * A, 4 * A, 5 * A, 6 * A, 64, 11 * A, kc, 8 * A, ks, vs,
                                          stream=0)

    def att(dims=d, ks=9 * A, vs=10 * A, kc=7 * A):
        return mi.mi_paged_decode_attention_fp8(dims, A, kc, 8 * A, ks, vs, 4 * A, 5 * A, 0.125, 11 * A, 12 * A,
                                                workspace_bytes=1 << 20, stream=0)
    for call in (app, att):
        assert call(ks=None) == mi.MI_ERR_INVALID_ARG
        assert call(vs=None) == mi.MI_ERR_INVALID_ARG
        assert call(kc=7 * A + 8) == mi.MI_ERR_INVALID_ARG
        assert call(dims=mi.dims(2, 4, 3, 64, 8, 4)) == mi.MI_ERR_UNSUPPORTED
        assert call(dims=mi.dims(0, 4, 2, 64, 8, 4)) == mi.MI_OK
    assert app(dims=mi.dims(2, 4, 2, 96, 8, 4)) == mi.MI_ERR_UNSUPPORTED


def test_token_slots_match_model_after_churn(mi):
    from workloads import PREFILL_WORKLOADS, prefill_setup_pool
    w = WORKLOADS["qwen3_8b"]
    order = initial_free_order(w)
    lib = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    model = PoolModel(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    ctx = context_lengths(w)
    setup_pool(w, lib, ctx)
    setup_pool(w, model, ctx)
    r = np.random.Generator(np.random.PCG64(11))
    for b in range(0, w.B, 5):
        n = int(ctx[b])
        first = int(r.integers(0, n))
        count = int(r.integers(0, n - first + 1))
        assert np.array_equal(lib.token_slots(b, first, count), model.token_slots(b, first, count))
    pw = PREFILL_WORKLOADS["prefill_small"]
    lib2 = mi.Pool(pw.num_blocks, pw.max_seqs, pw.max_blocks_per_seq, None)
    model2 = PoolModel(pw.num_blocks, pw.max_seqs, pw.max_blocks_per_seq, None)
    prefill_setup_pool(pw, lib2)
    prefill_setup_pool(pw, model2)
    h, m = pw.lengths()
    for b in range(pw.B):
        assert np.array_equal(lib2.token_slots(b, int(h[b]), int(m[b])),
                              model2.token_slots(b, int(h[b]), int(m[b])))


def test_token_slots_errors(mi):
    p = mi.Pool(8, 2, 4)
    assert p.alloc(0, 20) == 0
    st, _ = mi.mi_kv_pool_token_slots(p.handle, 1, 0, 1)
    assert st == mi.MI_ERR_UNKNOWN_SEQ
    assert mi.mi_kv_pool_token_slots(p.handle, 0, 15, 6)[0] == mi.MI_ERR_INVALID_ARG  # past token 20
    assert mi.mi_kv_pool_token_slots(p.handle, 0, -1, 2)[0] == mi.MI_ERR_INVALID_ARG
    st, s = mi.mi_kv_pool_token_slots(p.handle, 0, 14, 6)
    assert st == mi.MI_OK and len(s) == 6
    st, s = mi.mi_kv_pool_token_slots(p.handle, 0, 20, 0)
    assert st == mi.MI_OK and len(s) == 0


def test_prefill_rejects_bad_args_without_a_gpu(mi):
    d = mi.dims(2, 4, 2, 64, 8, 4)
    P = dict(q=16, k_cache=16, v_cache=16, block_tables=16, context_lens=16, query_start=16, scale=1.0,
             out=16, stream=0)
    odd = mi.dims(2, 4, 2, 96, 8, 4)
    assert mi.mi_paged_prefill_attention(odd, 4, 2, **P) == mi.MI_ERR_UNSUPPORTED
    wide = mi.dims(2, 18, 2, 64, 8, 4)  # G = 9
    assert mi.mi_paged_prefill_attention(wide, 4, 2, **P) == mi.MI_ERR_UNSUPPORTED
    assert mi.mi_paged_prefill_attention(d, -1, 2, **P) == mi.MI_ERR_INVALID_ARG
    assert mi.mi_paged_prefill_attention(d, 4, -2, **P) == mi.MI_ERR_INVALID_ARG
    assert mi.mi_paged_prefill_attention(d, 4, 2, **dict(P, scale=float("nan"))) == mi.MI_ERR_INVALID_ARG
    assert mi.mi_paged_prefill_attention(d, 4, 2, **dict(P, query_start=None)) == mi.MI_ERR_INVALID_ARG
    assert mi.mi_paged_prefill_attention(d, 4, 2, **dict(P, out=24)) == mi.MI_ERR_INVALID_ARG  # misaligned
    # nothing to do: no call reaches the GPU
    assert mi.mi_paged_prefill_attention(d, 0, 0, **dict(P, q=None, out=None)) == mi.MI_OK
    assert mi.mi_paged_prefill_attention(mi.dims(0, 4, 2, 64, 8, 4), 0, 0, **P) == mi.MI_OK
