"""GPU parity of mi_paged_kv_append against the oracle: bit-exact q_out and
cache contents, every byte the append must not touch left as it was (the
caches start filled with a NaN canary outside the live history)."""
import numpy as np
import pytest

import oracle
from helpers import from_dev_u16, grow, pools_for, to_dev_i32, to_dev_u16
from workloads import WORKLOADS, bf16_normal, device_fill_cache, history_cache, new_token_values

pytestmark = pytest.mark.gpu


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


@pytest.mark.parametrize("name,layers", [("tiny", [0]), ("qwen3_1p7b", [0]), ("skewed", [0]),
                                         ("qwen25_7b_sweep", [0, 27])])
def test_append_bit_exact(cuda_device, name, layers):
    import torch
    mi = _mi()
    w = WORKLOADS[name]
    lib, model, ctx = pools_for(w)
    bt_hist, _, _ = lib.batch_meta(range(w.B))
    grow(lib, w.B, ctx + 1)
    grow(model, w.B, ctx + 1)
    bt, cl, sl = lib.batch_meta(range(w.B))
    bt_m, cl_m, sl_m = model.batch_meta(range(w.B))
    assert np.array_equal(bt, bt_m) and np.array_equal(sl, sl_m)
    pos = (cl - 1).astype(np.int32)
    assert np.array_equal(oracle.slot_mapping(bt_m, pos), sl)
    st, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    assert st == 0
    table_ref = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    rope_d = torch.from_numpy(table).to(cuda_device)
    pos_d, sl_d = to_dev_i32(pos, cuda_device), to_dev_i32(sl, cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for layer in layers:
        kc, vc = history_cache(w, layer, bt_hist, ctx)
        q, k, v = new_token_values(w, layer)
        kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)
        q_d, k_d, v_d = (to_dev_u16(a, cuda_device) for a in (q, k, v))
        qo_d = torch.empty_like(q_d)
        assert mi.mi_paged_kv_append(d, q_d, k_d, v_d, pos_d, sl_d, rope_d, w.max_pos, qo_d, kc_d, vc_d,
                                     err) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        q_ref, st = oracle.append(q, k, v, pos, sl_m, table_ref, kc, vc)
        assert st == 0
        assert np.array_equal(from_dev_u16(qo_d), q_ref)
        assert np.array_equal(from_dev_u16(kc_d), kc)
        assert np.array_equal(from_dev_u16(vc_d), vc)


def test_append_in_place_q(cuda_device):
    import torch
    mi = _mi()
    w = WORKLOADS["tiny"]
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, sl = lib.batch_meta(range(w.B))
    pos = (cl - 1).astype(np.int32)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    q, k, v = new_token_values(w, 0)
    kc = np.zeros((w.num_blocks, w.Hkv, 16, w.head_dim), np.uint16)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    q_d = to_dev_u16(q, cuda_device)
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(kc, cuda_device)
    assert mi.mi_paged_kv_append(d, q_d, to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device),
                                 to_dev_i32(pos, cuda_device), to_dev_i32(sl, cuda_device),
                                 torch.from_numpy(table).to(cuda_device), w.max_pos, q_d, kc_d, vc_d) == 0
    torch.cuda.synchronize()
    q_ref, _ = oracle.append(q, k, v, pos, sl, oracle.rope_table(w.theta, w.head_dim, w.max_pos), kc, kc.copy())
    assert np.array_equal(from_dev_u16(q_d), q_ref)


def test_append_full_size_serving_layer(cuda_device):
    """Qwen3-8B-shaped layer at full size (24,576-block pool after churn): every
    written slot equals the oracle's rotation, nothing else in the 1.6 GB of
    cache changes."""
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_8b"]
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    grow(model, w.B, ctx + 1)
    bt, cl, sl = lib.batch_meta(range(w.B))
    assert np.array_equal(sl, model.batch_meta(range(w.B))[2])
    pos = (cl - 1).astype(np.int32)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    table_ref = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    shape = (w.num_blocks, w.Hkv, 16, w.head_dim)
    kc_d = torch.empty(shape, dtype=torch.bfloat16, device=cuda_device)
    vc_d = torch.empty_like(kc_d)
    device_fill_cache(w, 0, kc_d, vc_d)
    k0, v0 = kc_d.clone(), vc_d.clone()
    q, k, v = new_token_values(w, 0)
    q_d = to_dev_u16(q, cuda_device)
    qo_d = torch.empty_like(q_d)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    assert mi.mi_paged_kv_append(d, q_d, to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device),
                                 to_dev_i32(pos, cuda_device), to_dev_i32(sl, cuda_device),
                                 torch.from_numpy(table).to(cuda_device), w.max_pos, qo_d, kc_d, vc_d,
                                 err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    blk = torch.from_numpy((sl // 16).astype(np.int64)).to(cuda_device)
    off = torch.from_numpy((sl % 16).astype(np.int64)).to(cuda_device)
    got_k = from_dev_u16(kc_d[blk, :, off])  # [B][Hkv][d]
    got_v = from_dev_u16(vc_d[blk, :, off])
    for b in range(w.B):
        assert np.array_equal(got_k[b], oracle.rope_rotate(k[b], table_ref, int(pos[b])))
        assert np.array_equal(got_v[b], v[b])
        assert np.array_equal(from_dev_u16(qo_d[b]), oracle.rope_rotate(q[b], table_ref, int(pos[b])))
    kc_d[blk, :, off] = k0[blk, :, off]
    vc_d[blk, :, off] = v0[blk, :, off]
    assert torch.equal(kc_d.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(vc_d.view(torch.int16), v0.view(torch.int16))


def test_append_bad_slot_and_position_flagged(cuda_device):
    import torch
    mi = _mi()
    B, Hq, Hkv, dd, nb = 3, 4, 2, 64, 4
    r = np.random.Generator(np.random.PCG64(5))
    from workloads import bf16_normal
    q = bf16_normal(r, (B, Hq, dd)); k = bf16_normal(r, (B, Hkv, dd)); v = bf16_normal(r, (B, Hkv, dd))
    _, table = mi.mi_rope_table(1e6, dd, 8)
    kc = np.full((nb, Hkv, 16, dd), 0x1234, np.uint16)
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(kc, cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    d = mi.dims(B, Hq, Hkv, dd, nb, 4)
    pos = np.array([1, 9, 2], np.int32)          # 9 is past the table
    slots = np.array([5, 3, nb * 16], np.int32)  # nb*16 is past the cache
    qo_d = torch.zeros_like(to_dev_u16(q, cuda_device))
    assert mi.mi_paged_kv_append(d, to_dev_u16(q, cuda_device), to_dev_u16(k, cuda_device),
                                 to_dev_u16(v, cuda_device), to_dev_i32(pos, cuda_device),
                                 to_dev_i32(slots, cuda_device), torch.from_numpy(table).to(cuda_device), 8,
                                 qo_d, kc_d, vc_d, err) == 0
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & mi.MI_DEVERR_BAD_POS and e & mi.MI_DEVERR_BAD_SLOT
    # request 0 was written, request 1 (bad position) and 2's cache (bad slot) were not
    kc_ref = kc.copy()
    kc_ref[0, :, 5] = oracle.rope_rotate(k[0], oracle.rope_table(1e6, dd, 8), 1)
    assert np.array_equal(from_dev_u16(kc_d), kc_ref)


def test_append_bit_exact_on_extreme_values(cuda_device):
    """Finite bf16 inputs over the whole exponent range (subnormals, signed
    zeros, values near the largest finite bf16, pairs that nearly cancel)
    rotate to the oracle's bits."""
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(77))
    B, Hq, Hkv, dd, nb, max_pos = 16, 8, 2, 128, 4, 4096
    n = B * (Hq + 2 * Hkv) * dd
    sign = r.integers(0, 2, n).astype(np.uint16) << 15
    expo = r.integers(0, 255, n).astype(np.uint16)      # 0 = zero/subnormal, 254 = largest finite binade
    mant = r.integers(0, 128, n).astype(np.uint16)
    bits = (sign | (expo << 7) | mant).astype(np.uint16)
    bits[: n // 8] &= 0x807F                              # a block of subnormals and signed zeros
    q = bits[: B * Hq * dd].reshape(B, Hq, dd).copy()
    k = bits[B * Hq * dd: B * (Hq + Hkv) * dd].reshape(B, Hkv, dd).copy()
    v = bits[B * (Hq + Hkv) * dd:].reshape(B, Hkv, dd).copy()
    k[0, 0, : dd // 2] = k[0, 0, dd // 2:]                # x1 == x2: the rotation nearly cancels
    pos = r.integers(0, max_pos, B).astype(np.int32)
    slots = (r.permutation(nb * 16)[:B]).astype(np.int32)
    st, table = mi.mi_rope_table(1e6, dd, max_pos)
    assert st == 0
    kc = np.full((nb, Hkv, 16, dd), 0x7FA5, np.uint16)
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(kc, cuda_device)
    qo_d = torch.empty((B, Hq, dd), dtype=torch.bfloat16, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    d = mi.dims(B, Hq, Hkv, dd, nb, 1)
    assert mi.mi_paged_kv_append(d, to_dev_u16(q, cuda_device), to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device),
                                 to_dev_i32(pos, cuda_device), to_dev_i32(slots, cuda_device),
                                 torch.from_numpy(table).to(cuda_device), max_pos, qo_d, kc_d, vc_d, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc_ref, vc_ref = kc.copy(), kc.copy()
    q_ref, st = oracle.append(q, k, v, pos, slots, oracle.rope_table(1e6, dd, max_pos), kc_ref, vc_ref)
    assert st == 0
    assert np.array_equal(from_dev_u16(qo_d), q_ref)
    assert np.array_equal(from_dev_u16(kc_d), kc_ref)
    assert np.array_equal(from_dev_u16(vc_d), vc_ref)


@pytest.mark.parametrize("B,d", [(4096, 128), (256, 128), (200, 64)])
def test_append_rotation_bit_exact_on_wide_values(cuda_device, B, d):
    """Rows of q (32 heads) and k (8 heads) at positions spread over a 32k
    table, values over many binades (with zeros of both signs and the bf16
    extremes): every rotated output equals the oracle's bit for bit,
    whichever internal route (single precision with exact transforms, or
    double) a kernel thread takes. 4,096 rows run the eight-pairs-per-thread
    kernel, a few hundred the two-pairs one."""
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(31 + B + d))
    Hq, Hkv, max_pos, nb = 32, 8, 32768, 300
    def wide(shape):
        x = r.standard_normal(shape) * 2.0 ** r.integers(-40, 40, shape)
        x[r.random(shape) < 0.01] = 0.0
        x[r.random(shape) < 0.01] = -0.0
        x[r.random(shape) < 0.001] = 3.3e38
        x[r.random(shape) < 0.001] = -1e-38
        return oracle.f64_to_bf16(x)
    q, k, v = wide((B, Hq, d)), wide((B, Hkv, d)), wide((B, Hkv, d))
    pos = r.integers(0, max_pos, B).astype(np.int32)
    slots = r.permutation(nb * 16)[:B].astype(np.int32)
    _, table = mi.mi_rope_table(1e6, d, max_pos)
    table_ref = oracle.rope_table(1e6, d, max_pos)
    kc = np.zeros((nb, Hkv, 16, d), np.uint16)
    vc = kc.copy()
    dm = mi.dims(B, Hq, Hkv, d, nb, 1)
    q_d = to_dev_u16(q, cuda_device)
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    qo_d = torch.empty_like(q_d)
    assert mi.mi_paged_kv_append(dm, q_d, to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device),
                                 to_dev_i32(pos, cuda_device), to_dev_i32(slots, cuda_device),
                                 torch.from_numpy(table).to(cuda_device), max_pos, qo_d, kc_d, vc_d, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q_ref, st = oracle.append(q, k, v, pos, slots, table_ref, kc, vc)
    assert st == 0
    assert np.array_equal(from_dev_u16(qo_d), q_ref)
    assert np.array_equal(from_dev_u16(kc_d), kc)
    assert np.array_equal(from_dev_u16(vc_d), vc)


NEAR_TIE_POSITIONS = [1, 3, 17, 100, 255, 1000, 2047, 4095]


@pytest.fixture(scope="module")
def near_tie_sets():
    """Near-tie rotation pairs for every table entry of the positions above
    (d = 128, theta = 1e6), from the oracle's table."""
    from near_ties import near_tie_sets as sets_for
    table = oracle.rope_table(1e6, 128, 4096)
    return table, sets_for(table, NEAR_TIE_POSITIONS, seed=2024)


@pytest.mark.parametrize("rows_per_position", [3, 40])  # 24 rows: two pairs per thread; 320: eight
def test_append_bit_exact_at_near_ties(cuda_device, near_tie_sets, rows_per_position):
    """Every rotation pair of every q and k head holds a pair whose exact
    rotated value lies within 4 fp32 ulps of a bf16 rounding midpoint or of
    a power of two (over 10^4 distinct such pairs): the places where a
    single-precision rotation could round differently. q_out and the cache
    rows equal the oracle's bit for bit through both thread layouts of the
    append (decode-sized and prefill-sized batches)."""
    import torch
    from near_ties import near_tie_rows
    mi = _mi()
    table_ref, sets = near_tie_sets
    Hq, Hkv, dh = 8, 2, 128
    rows, pos, distinct, kinds = near_tie_rows(sets, NEAR_TIE_POSITIONS, rows_per_position, Hq + Hkv)
    assert distinct >= 10_000 and kinds[0] > 0 and kinds[1] > 0, (distinct, kinds)
    B = rows.shape[0]
    q, k = np.ascontiguousarray(rows[:, :Hq]), np.ascontiguousarray(rows[:, Hq:])
    v = bf16_normal(np.random.Generator(np.random.PCG64(11)), (B, Hkv, dh))
    nb = B
    sl = (np.arange(B) * 16 + np.arange(B) % 16).astype(np.int32)  # block b, a different row in each
    kc = np.full((nb, Hkv, 16, dh), 0x7FA5, np.uint16)
    vc = kc.copy()
    _, table = mi.mi_rope_table(1e6, dh, 4096)
    assert np.array_equal(table, table_ref)
    d = mi.dims(B, Hq, Hkv, dh, nb, 1)
    q_d = to_dev_u16(q, cuda_device)
    qo_d = torch.empty_like(q_d)
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    assert mi.mi_paged_kv_append(d, q_d, to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device),
                                 to_dev_i32(pos, cuda_device), to_dev_i32(sl, cuda_device),
                                 torch.from_numpy(table).to(cuda_device), 4096, qo_d, kc_d, vc_d, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q_ref, st = oracle.append(q, k, v, pos, sl, table_ref, kc, vc)
    assert st == 0
    assert np.array_equal(from_dev_u16(qo_d), q_ref)
    assert np.array_equal(from_dev_u16(kc_d), kc)
    assert np.array_equal(from_dev_u16(vc_d), vc)


def test_step_bit_exact_at_near_ties(cuda_device, near_tie_sets):
    """The fused decode step rotates q and the new k with the same exact
    rule: on near-tie inputs its q_out and the new cache rows equal the
    oracle's append bit for bit (the attention output is not compared here:
    the near-tie values span 2^-30 .. 2^30)."""
    import torch
    from near_ties import near_tie_rows
    mi = _mi()
    table_ref, sets = near_tie_sets
    Hq, Hkv, dh = 8, 2, 128
    rows, pos, distinct, _ = near_tie_rows(sets, NEAR_TIE_POSITIONS, 3, Hq + Hkv)
    B = rows.shape[0]
    q, k = np.ascontiguousarray(rows[:, :Hq]), np.ascontiguousarray(rows[:, Hq:])
    r = np.random.Generator(np.random.PCG64(12))
    v = bf16_normal(r, (B, Hkv, dh))
    cl = (pos + 1).astype(np.int32)            # the new token sits at position cl - 1
    nblk = -(-cl // 16)
    nb = int(nblk.sum())
    mbps = int(nblk.max())
    perm = r.permutation(nb)
    bt = np.full((B, mbps), -1, np.int32)
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    kc = bf16_normal(r, (nb, Hkv, 16, dh))
    vc = bf16_normal(r, (nb, Hkv, 16, dh))
    _, table = mi.mi_rope_table(1e6, dh, 4096)
    d = mi.dims(B, Hq, Hkv, dh, nb, mbps)
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=cuda_device)
    q_d = to_dev_u16(q, cuda_device)
    qo_d, out = torch.empty_like(q_d), torch.empty_like(q_d)
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    assert mi.mi_paged_decode_step(d, q_d, to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device),
                                   torch.from_numpy(table).to(cuda_device), 4096, to_dev_i32(bt, cuda_device),
                                   to_dev_i32(cl, cuda_device), 1.0 / np.sqrt(dh), qo_d, kc_d, vc_d, out, ws,
                                   dev_err=err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q_ref, st = oracle.append(q, k, v, pos, oracle.slot_mapping(bt, pos), table_ref, kc, vc)
    assert st == 0
    assert np.array_equal(from_dev_u16(qo_d), q_ref)
    assert np.array_equal(from_dev_u16(kc_d), kc)
    assert np.array_equal(from_dev_u16(vc_d), vc)
