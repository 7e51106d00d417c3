"""GPU parity of mi_paged_decode_attention against the fp64 oracle.

Tolerance (bf16 inputs, unit-variance V): max |gpu - oracle| <= 1e-2 and mean
|gpu - oracle| <= 1e-3 over all outputs. Covered: the small workloads in full,
the Qwen3-8B-shaped serving layer at full size (every request and head), the
Qwen2.5-7B 128-step sweep at checkpoints, both kernel variants, several grid
sizes (split counts), edge context lengths with NaN in unused slots, exact
closed forms (one-token context returns V), bitwise paging invariance, zero
rows for empty contexts, and the device error word for bad tables.
"""
import numpy as np
import pytest

import oracle
from helpers import (assert_attention_close, from_dev_u16, gather_used_blocks, grow, pools_for, to_dev_i32,
                     to_dev_u16)
from workloads import (BLOCK, CANARY_BF16, WORKLOADS, bf16_normal, device_fill_cache, history_cache,
                       new_token_values)

pytestmark = pytest.mark.gpu
VARIANTS = [1, 2]  # MI_ATTN_MMA, MI_ATTN_FMA


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


def _workspace(mi, d, device):
    import torch
    n = mi.mi_paged_decode_workspace_bytes(d)
    assert n > 0
    return torch.empty(n // 4 + 4, dtype=torch.float32, device=device)


def _run(mi, d, q_d, kc_d, vc_d, bt_d, cl_d, scale, ws, variant, ctas, device):
    import torch
    out = torch.full(q_d.shape, float("nan"), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    st = mi.mi_paged_decode_attention_variant(d, q_d, kc_d, vc_d, bt_d, cl_d, scale, out, ws,
                                              variant=variant, ctas=ctas, dev_err=err)
    assert st == 0, mi.status_string(st)
    torch.cuda.synchronize()
    return from_dev_u16(out), int(err.item())


def _small_case(name, device):
    """History + one appended token (through the library), on the device."""
    import torch
    mi = _mi()
    w = WORKLOADS[name]
    lib, model, ctx = pools_for(w)
    bt_hist, _, _ = lib.batch_meta(range(w.B))
    grow(lib, w.B, ctx + 1)
    grow(model, w.B, ctx + 1)
    bt, cl, sl = lib.batch_meta(range(w.B))
    kc, vc = history_cache(w, 0, bt_hist, ctx)
    q, k, v = new_token_values(w, 0)
    pos = (cl - 1).astype(np.int32)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    kc_d, vc_d = to_dev_u16(kc, device), to_dev_u16(vc, device)
    q_d = to_dev_u16(q, device)
    assert mi.mi_paged_kv_append(d, q_d, to_dev_u16(k, device), to_dev_u16(v, device), to_dev_i32(pos, device),
                                 to_dev_i32(sl, device), torch.from_numpy(table).to(device), w.max_pos, q_d,
                                 kc_d, vc_d) == 0
    torch.cuda.synchronize()
    # oracle inputs: its own append of the same token on its own table copy
    q_ref, st = oracle.append(q, k, v, pos, model.batch_meta(range(w.B))[2],
                              oracle.rope_table(w.theta, w.head_dim, w.max_pos), kc, vc)
    assert st == 0
    return w, d, q_ref, kc, vc, bt, cl, q_d, kc_d, vc_d


@pytest.mark.parametrize("name", ["tiny", "qwen3_1p7b", "skewed"])
def test_attention_matches_oracle(cuda_device, name):
    mi = _mi()
    w, d, q, kc, vc, bt, cl, q_d, kc_d, vc_d = _small_case(name, cuda_device)
    ref = oracle.paged_attention(q, kc, vc, bt, cl, w.scale, nthreads=8)
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(cl, cuda_device)
    ws = _workspace(mi, d, cuda_device)
    outs = {}
    for var in VARIANTS:
        for ctas in (0, 1, 7):
            out, err = _run(mi, d, q_d, kc_d, vc_d, bt_d, cl_d, w.scale, ws, var, ctas, cuda_device)
            assert err == 0
            assert_attention_close(out, ref, f"{name} variant {var} ctas {ctas}")
            outs[(var, ctas)] = out
    # the default entry point is the MMA variant on the persistent grid
    import torch
    out = torch.empty_like(q_d)
    assert mi.mi_paged_decode_attention(d, q_d, kc_d, vc_d, bt_d, cl_d, w.scale, out, ws) == 0
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_u16(out), outs[(1, 0)])


def test_attention_full_size_serving_layer(cuda_device):
    """Qwen3-8B-shaped layer at full size (B = 64, contexts up to 8k, churned
    24,576-block pool), persistent grid as timed by the benchmark: every
    request and every head against the oracle."""
    import os
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_8b"]
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, sl = lib.batch_meta(range(w.B))
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    kc_d = torch.empty(shape, dtype=torch.bfloat16, device=cuda_device)
    vc_d = torch.empty_like(kc_d)
    device_fill_cache(w, 0, kc_d, vc_d)
    q, _, _ = new_token_values(w, 0)
    q_d = to_dev_u16(q, cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    ws = _workspace(mi, d, cuda_device)
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(cl, cuda_device)
    # every request's blocks, renumbered into a host cache the oracle walks
    kc_s, vc_s, bt_s, _ = gather_used_blocks(kc_d, vc_d, bt, cl)
    ref = oracle.paged_attention(q, kc_s, vc_s, bt_s, cl, w.scale, nthreads=os.cpu_count() or 8)
    for var in VARIANTS:
        out, err = _run(mi, d, q_d, kc_d, vc_d, bt_d, cl_d, w.scale, ws, var, 0, cuda_device)
        assert err == 0
        assert_attention_close(out, ref, f"qwen3_8b variant {var}")


def test_attention_sweep_checkpoints(cuda_device):
    """Qwen2.5-7B-shaped sweep: 128 decode steps over 28 layers through the
    library (pool growth, append, attention). The oracle follows layers 0 and
    27 with its own pool copy and appends, and checks attention at several
    steps and the final caches bit for bit."""
    import torch
    mi = _mi()
    w = WORKLOADS["qwen25_7b_sweep"]
    lib, model, ctx = pools_for(w)
    bt_hist, _, _ = lib.batch_meta(range(w.B))
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    table_ref = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    rope_d = torch.from_numpy(table).to(cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    ws = _workspace(mi, d, cuda_device)
    follow = (0, 27)
    host = {}
    caches = []
    for layer in range(w.layers):
        kc, vc = history_cache(w, layer, bt_hist, ctx)
        caches.append((to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)))
        if layer in follow:
            host[layer] = (kc, vc)
    checkpoints = {0, 1, 15, 16, 63, 127}
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for step in range(w.sweep_steps):
        grow(lib, w.B, ctx + step + 1)
        grow(model, w.B, ctx + step + 1)
        bt, cl, sl = lib.batch_meta(range(w.B))
        bt_m, cl_m, sl_m = model.batch_meta(range(w.B))
        assert np.array_equal(bt, bt_m) and np.array_equal(sl, sl_m)
        pos = (cl - 1).astype(np.int32)
        bt_d, cl_d, sl_d, pos_d = (to_dev_i32(a, cuda_device) for a in (bt, cl, sl, pos))
        for layer in range(w.layers):
            q, k, v = new_token_values(w, layer, step)
            q_d = to_dev_u16(q, cuda_device)
            kc_d, vc_d = caches[layer]
            assert mi.mi_paged_kv_append(d, q_d, to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device), pos_d,
                                         sl_d, rope_d, w.max_pos, q_d, kc_d, vc_d, err) == 0
            out = torch.empty_like(q_d)
            assert mi.mi_paged_decode_attention(d, q_d, kc_d, vc_d, bt_d, cl_d, w.scale, out, ws, dev_err=err) == 0
            if layer in follow:
                kc, vc = host[layer]
                q_ref, st = oracle.append(q, k, v, pos, sl_m, table_ref, kc, vc)
                assert st == 0
                if step in checkpoints:
                    torch.cuda.synchronize()
                    assert np.array_equal(from_dev_u16(q_d), q_ref)
                    ref = oracle.paged_attention(q_ref, kc, vc, bt_m, cl_m, w.scale, nthreads=8)
                    assert_attention_close(from_dev_u16(out), ref, f"sweep step {step} layer {layer}")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for layer in follow:
        assert np.array_equal(from_dev_u16(caches[layer][0]), host[layer][0])
        assert np.array_equal(from_dev_u16(caches[layer][1]), host[layer][1])


def _edge_case(device, d_head, lens, Hq=8, Hkv=2, seed=77, extra_blocks=9):
    """Random paged cache for the given post-append lengths, NaN canary in
    every slot past a request's length and in unused blocks."""
    r = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(lens, np.int32)
    nblk = [-(-max(int(n), 0) // BLOCK) for n in lens]
    nb = sum(nblk) + extra_blocks
    perm = r.permutation(nb)
    mbps = max(max(nblk), 1)
    bt = np.full((len(lens), mbps), -1, np.int32)
    kc = np.full((nb, Hkv, BLOCK, d_head), CANARY_BF16, np.uint16)
    vc = kc.copy()
    i = 0
    for b, n in enumerate(lens):
        for j in range(nblk[b]):
            blk = int(perm[i]); i += 1
            bt[b, j] = blk
            m = min(BLOCK, int(n) - j * BLOCK)
            kc[blk, :, :m] = bf16_normal(r, (Hkv, m, d_head))
            vc[blk, :, :m] = bf16_normal(r, (Hkv, m, d_head))
    q = bf16_normal(r, (len(lens), Hq, d_head))
    return q, kc, vc, bt, lens, mbps, nb


EDGE_LENS = [1, 15, 16, 17, 31, 32, 33, 0, 255, 256, 257, 4097, 2, 48, -3, 1000]


@pytest.mark.parametrize("d_head,Hq,Hkv", [(128, 8, 2), (64, 4, 2), (128, 7, 1), (128, 8, 8), (128, 16, 2)])
def test_attention_edge_lengths(cuda_device, d_head, Hq, Hkv):
    mi = _mi()
    q, kc, vc, bt, lens, mbps, nb = _edge_case(cuda_device, d_head, EDGE_LENS, Hq, Hkv)
    scale = 1.0 / np.sqrt(d_head)
    ref = oracle.paged_attention(q, kc, vc, bt, lens, scale, nthreads=8)
    d = mi.dims(len(lens), Hq, Hkv, d_head, nb, mbps)
    q_d, kc_d, vc_d = (to_dev_u16(a, cuda_device) for a in (q, kc, vc))
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(lens, cuda_device)
    ws = _workspace(mi, d, cuda_device)
    for var in VARIANTS:
        for ctas in (0, 1, 2, 3, 13, 100):
            out, err = _run(mi, d, q_d, kc_d, vc_d, bt_d, cl_d, scale, ws, var, ctas, cuda_device)
            assert err == 0
            assert_attention_close(out, ref, f"edge d{d_head} G{Hq // Hkv} var {var} ctas {ctas}")
            empty = lens <= 0
            assert np.all(out[empty] == 0)


def test_attention_growing_scores(cuda_device):
    """Keys whose magnitude grows along the context (block j scaled by
    1 + j / 2): each row's max moves by far more than 2^8 (base 2) from block
    to block, and at small grids the split-KV pieces merged at the end carry
    very different maxima. Rows are nearly one-hot, so outputs are as large
    as V; the bound is the bf16 rounding of each weight and of the output
    (2^-9 relative each, factor 2 margin): |got - ref| <= 2^-8 (sum_i p_i
    |v_i| + |ref|), sum_i p_i |v_i| being the oracle's attention over |V|."""
    mi = _mi()
    q, kc, vc, bt, lens, mbps, nb = _edge_case(cuda_device, 128, [1500, 700, 33, 4000], Hq=8, Hkv=2)
    k64 = oracle.bf16_to_f64(kc)
    for b in range(len(lens)):
        for j in range(-(-int(lens[b]) // BLOCK)):
            k64[bt[b, j]] *= 1.0 + j / 2.0
    kc = oracle.f64_to_bf16(k64)
    scale = 1.0 / np.sqrt(128)
    ref = oracle.paged_attention(q, kc, vc, bt, lens, scale, nthreads=8)
    vabs = np.where(np.isnan(oracle.bf16_to_f64(vc)), vc, vc & np.uint16(0x7FFF)).astype(np.uint16)
    ref_abs = oracle.paged_attention(q, kc, vabs, bt, lens, scale, nthreads=8)
    bound = 2.0 ** -8 * (ref_abs + np.abs(ref))
    d = mi.dims(len(lens), 8, 2, 128, nb, mbps)
    q_d, kc_d, vc_d = (to_dev_u16(a, cuda_device) for a in (q, kc, vc))
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(lens, cuda_device)
    ws = _workspace(mi, d, cuda_device)
    for var in VARIANTS:
        for ctas in (0, 1, 3, 13, 100):
            out, err = _run(mi, d, q_d, kc_d, vc_d, bt_d, cl_d, scale, ws, var, ctas, cuda_device)
            assert err == 0
            g = oracle.bf16_to_f64(out)
            assert np.all(np.isfinite(g))
            worst = float(np.max(np.abs(g - ref) / bound))
            assert worst <= 1.0, f"var {var} ctas {ctas}: error {worst:.2f} x the bound"


def test_one_token_context_returns_v_exactly(cuda_device):
    mi = _mi()
    q, kc, vc, bt, lens, mbps, nb = _edge_case(cuda_device, 128, [1, 1, 1], Hq=8, Hkv=2)
    d = mi.dims(3, 8, 2, 128, nb, mbps)
    q_d, kc_d, vc_d = (to_dev_u16(a, cuda_device) for a in (q, kc, vc))
    ws = _workspace(mi, d, cuda_device)
    for var in VARIANTS:
        out, err = _run(mi, d, q_d, kc_d, vc_d, to_dev_i32(bt, cuda_device), to_dev_i32(lens, cuda_device),
                        0.0883883, ws, var, 0, cuda_device)
        for b in range(3):
            for j in range(8):
                assert np.array_equal(out[b, j], vc[bt[b, 0], j // 4, 0])


def test_paging_invariance_bitwise(cuda_device):
    import torch
    mi = _mi()
    q, kc, vc, bt, lens, mbps, nb = _edge_case(cuda_device, 128, [300, 17, 1, 999, 64], Hq=8, Hkv=2)
    d = mi.dims(len(lens), 8, 2, 128, nb, mbps)
    ws = _workspace(mi, d, cuda_device)
    perm = np.random.Generator(np.random.PCG64(9)).permutation(nb)
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    for var in VARIANTS:
        for ctas in (0, 3):
            a, _ = _run(mi, d, *(to_dev_u16(x, cuda_device) for x in (q, kc, vc)), to_dev_i32(bt, cuda_device),
                        to_dev_i32(lens, cuda_device), 0.088, ws, var, ctas, cuda_device)
            b, _ = _run(mi, d, *(to_dev_u16(x, cuda_device) for x in (q, kc2, vc2)), to_dev_i32(bt2, cuda_device),
                        to_dev_i32(lens, cuda_device), 0.088, ws, var, ctas, cuda_device)
            assert np.array_equal(a, b)


def test_bad_table_and_context_set_error_bits(cuda_device):
    mi = _mi()
    q, kc, vc, bt, lens, mbps, nb = _edge_case(cuda_device, 128, [40, 20, 33], Hq=8, Hkv=2)
    bt = bt.copy()
    bt[1, 0] = nb + 1000   # block id past the cache
    lens = lens.copy()
    lens[2] = mbps * BLOCK + 5  # longer than a table row
    d = mi.dims(3, 8, 2, 128, nb, mbps)
    ws = _workspace(mi, d, cuda_device)
    for var in VARIANTS:
        out, err = _run(mi, d, *(to_dev_u16(x, cuda_device) for x in (q, kc, vc)), to_dev_i32(bt, cuda_device),
                        to_dev_i32(lens, cuda_device), 0.088, ws, var, 0, cuda_device)
        assert err & mi.MI_DEVERR_BAD_BLOCK and err & mi.MI_DEVERR_BAD_CONTEXT
        # request 0 is untouched by the faults
        ref = oracle.paged_attention(q[:1], kc, vc, bt[:1], lens[:1], 0.088)
        assert_attention_close(out[:1], ref, "request 0 next to bad entries")


def test_workspace_too_small_is_rejected(cuda_device):
    import torch
    mi = _mi()
    d = mi.dims(2, 8, 2, 128, 8, 4)
    n = mi.mi_paged_decode_workspace_bytes(d)
    ws = torch.empty(n // 4, dtype=torch.float32, device=cuda_device)
    z = torch.zeros(16, dtype=torch.int32, device=cuda_device)
    st = mi.mi_paged_decode_attention(d, z, z, z, z, z, 1.0, z, ws, workspace_bytes=n - 16)
    assert st == mi.MI_ERR_INVALID_ARG

