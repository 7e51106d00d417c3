"""GPU parity of mi_paged_decode_step, the fused append + attention of one
layer: its q_out, the new cache rows and the attention output carry the same
bits as mi_paged_kv_append followed by mi_paged_decode_attention (both pinned
to the oracle elsewhere), and the output is within the attention tolerance of
the fp64 oracle's append + attention. Covered: the small workloads in full,
the Qwen3-8B-shaped serving layer at full size (every request and head
against the oracle), edge context lengths, head
dims 64 and 128 and several GQA groups, NaN in unused cache rows, a position
past the RoPE table, the overlap check on q / q_out, and early start
(MI_STEP_EARLY_START) over a stack of layers, eager and graph-replayed."""
import numpy as np
import pytest

import oracle
from helpers import (assert_attention_close, from_dev_u16, gather_used_blocks, grow, pools_for, to_dev_i32,
                     to_dev_u16)
from workloads import BLOCK, WORKLOADS, bf16_normal, device_fill_cache, history_cache, new_token_values

pytestmark = pytest.mark.gpu


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


def _both(device, d, q, k, v, table, max_pos, bt, cl, kc, vc, scale):
    """(two-call results, fused results): each (q_out, k_cache, v_cache, out,
    err) on fresh device copies of the same inputs."""
    import torch
    mi = _mi()
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=device)
    tab_d = torch.from_numpy(table).to(device)
    bt_d, cl_d = to_dev_i32(bt, device), to_dev_i32(cl, device)
    pos = (cl - 1).astype(np.int32)
    sl = np.array([bt[b, (cl[b] - 1) // 16] * 16 + (cl[b] - 1) % 16 for b in range(len(cl))], np.int32)
    res = []
    for fused in (False, True):
        q_d, k_d, v_d = to_dev_u16(q, device), to_dev_u16(k, device), to_dev_u16(v, device)
        kc_d, vc_d = to_dev_u16(kc, device), to_dev_u16(vc, device)
        qo_d = torch.full_like(q_d, float("nan"))
        out = torch.full_like(q_d, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=device)
        if fused:
            st = mi.mi_paged_decode_step(d, q_d, k_d, v_d, tab_d, max_pos, bt_d, cl_d, scale, qo_d, kc_d, vc_d,
                                         out, ws, dev_err=err)
            assert st == 0, mi.status_string(st)
        else:
            assert mi.mi_paged_kv_append(d, q_d, k_d, v_d, to_dev_i32(pos, device), to_dev_i32(sl, device), tab_d,
                                         max_pos, qo_d, kc_d, vc_d, err) == 0
            assert mi.mi_paged_decode_attention(d, qo_d, kc_d, vc_d, bt_d, cl_d, scale, out, ws, dev_err=err) == 0
        torch.cuda.synchronize()
        res.append((from_dev_u16(qo_d), from_dev_u16(kc_d), from_dev_u16(vc_d), from_dev_u16(out),
                    int(err.item())))
    return res


def _assert_same(two, fused):
    for i, what in enumerate(("q_out", "k_cache", "v_cache", "out")):
        assert np.array_equal(two[i], fused[i]), f"{what} differs from the two-call path"
    assert two[4] == fused[4] == 0


@pytest.mark.parametrize("name", ["tiny", "qwen3_1p7b", "skewed"])
def test_step_matches_two_calls_and_oracle(cuda_device, name):
    mi = _mi()
    w = WORKLOADS[name]
    lib, model, ctx = pools_for(w)
    bt_hist, _, _ = lib.batch_meta(range(w.B))
    grow(lib, w.B, ctx + 1)
    grow(model, w.B, ctx + 1)
    bt, cl, sl = lib.batch_meta(range(w.B))
    kc, vc = history_cache(w, 0, bt_hist, ctx)
    q, k, v = new_token_values(w, 0)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    two, fused = _both(cuda_device, d, q, k, v, table, w.max_pos, bt, cl, kc, vc, w.scale)
    _assert_same(two, fused)
    # the oracle's own append + attention
    q_ref, st = oracle.append(q, k, v, (cl - 1).astype(np.int32), model.batch_meta(range(w.B))[2],
                              oracle.rope_table(w.theta, w.head_dim, w.max_pos), kc, vc)
    assert st == 0
    assert np.array_equal(fused[0], q_ref)
    assert np.array_equal(fused[1], kc) and np.array_equal(fused[2], vc)
    ref = oracle.paged_attention(q_ref, kc, vc, bt, cl, w.scale, nthreads=8)
    assert_attention_close(fused[3], ref, f"{name} fused step")


def test_step_full_size_serving_layer(cuda_device):
    """Qwen3-8B serving layer (B = 64, contexts up to 8k, fragmented pool,
    device-filled caches), in the launch configuration the benchmark times:
    the fused step equals the two calls bit for bit (q_out, both whole
    caches, the output), and equals the oracle's own append (q_out and every
    cache block the requests use, bit for bit) followed by its attention
    (every request and head, within the tolerance)."""
    import os
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_8b"]
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    kc0 = torch.empty(shape, dtype=torch.bfloat16, device=cuda_device)
    vc0 = torch.empty_like(kc0)
    device_fill_cache(w, 0, kc0, vc0)
    q, k, v = new_token_values(w, 0)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    tab_d = torch.from_numpy(table).to(cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=cuda_device)
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(cl, cuda_device)
    q_d, k_d, v_d = (to_dev_u16(a, cuda_device) for a in (q, k, v))
    pos = (cl - 1).astype(np.int32)
    sl = np.array([bt[b, (cl[b] - 1) // 16] * 16 + (cl[b] - 1) % 16 for b in range(w.B)], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    # the oracle's inputs: every block the requests use, before the step
    kc_s, vc_s, bt_s, used = gather_used_blocks(kc0, vc0, bt, cl)
    # two calls
    kc_a, vc_a = kc0.clone(), vc0.clone()
    qo_a, out_a = torch.empty_like(q_d), torch.empty_like(q_d)
    assert mi.mi_paged_kv_append(d, q_d, k_d, v_d, to_dev_i32(pos, cuda_device), to_dev_i32(sl, cuda_device), tab_d,
                                 w.max_pos, qo_a, kc_a, vc_a, err) == 0
    assert mi.mi_paged_decode_attention(d, qo_a, kc_a, vc_a, bt_d, cl_d, w.scale, out_a, ws, dev_err=err) == 0
    # fused, on the original caches
    qo_b, out_b = torch.empty_like(q_d), torch.empty_like(q_d)
    assert mi.mi_paged_decode_step(d, q_d, k_d, v_d, tab_d, w.max_pos, bt_d, cl_d, w.scale, qo_b, kc0, vc0, out_b,
                                   ws, dev_err=err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(qo_a.view(torch.int16), qo_b.view(torch.int16))
    assert torch.equal(kc_a.view(torch.int16), kc0.view(torch.int16))
    assert torch.equal(vc_a.view(torch.int16), vc0.view(torch.int16))
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    # the oracle's append (slots from its own slot mapping over the renumbered
    # tables) and attention over the same blocks
    q_ref, st = oracle.append(q, k, v, pos, oracle.slot_mapping(bt_s, pos),
                              oracle.rope_table(w.theta, w.head_dim, w.max_pos), kc_s, vc_s)
    assert st == 0
    assert np.array_equal(from_dev_u16(qo_b), q_ref)
    kc_f, vc_f, _, used_f = gather_used_blocks(kc0, vc0, bt, cl)
    assert used_f == used
    assert np.array_equal(kc_f, kc_s) and np.array_equal(vc_f, vc_s)
    ref = oracle.paged_attention(q_ref, kc_s, vc_s, bt_s, cl, w.scale, nthreads=os.cpu_count() or 8)
    assert_attention_close(from_dev_u16(out_b), ref, "qwen3_8b fused step")


@pytest.mark.parametrize("d_head,Hq,Hkv", [(128, 8, 2), (64, 4, 2), (128, 7, 1), (64, 8, 8), (128, 16, 2)])
def test_step_edge_lengths(cuda_device, d_head, Hq, Hkv):
    """Contexts of 1, 15, 16, 17, 31, 32, 33 and 200 tokens after the append
    (the new token first, last or alone in its block), NaN in every unused
    cache row, blocks scattered through the pool."""
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(d_head * 100 + Hq * 10 + Hkv))
    cl = np.array([1, 15, 16, 17, 31, 32, 33, 200], np.int32)
    B = len(cl)
    nblk = -(-cl // 16)
    nb = int(nblk.sum()) + 7
    mbps = int(nblk.max())
    perm = r.permutation(nb)
    bt = np.full((B, mbps), -1, np.int32)
    i = 0
    for b in range(B):
        for j in range(nblk[b]):
            bt[b, j] = perm[i]
            i += 1
    kc = np.full((nb, Hkv, 16, d_head), 0x7FA5, np.uint16)
    vc = kc.copy()
    for b in range(B):
        for t in range(cl[b] - 1):  # history; the step writes row cl - 1
            kc[bt[b, t // 16], :, t % 16] = bf16_normal(r, (Hkv, d_head))
            vc[bt[b, t // 16], :, t % 16] = bf16_normal(r, (Hkv, d_head))
    q, k, v = bf16_normal(r, (B, Hq, d_head)), bf16_normal(r, (B, Hkv, d_head)), bf16_normal(r, (B, Hkv, d_head))
    max_pos = 256
    _, table = mi.mi_rope_table(1e6, d_head, max_pos)
    d = mi.dims(B, Hq, Hkv, d_head, nb, mbps)
    scale = 1.0 / np.sqrt(d_head)
    two, fused = _both(cuda_device, d, q, k, v, table, max_pos, bt, cl, kc, vc, scale)
    _assert_same(two, fused)
    sl = np.array([bt[b, (cl[b] - 1) // 16] * 16 + (cl[b] - 1) % 16 for b in range(B)], np.int32)
    q_ref, st = oracle.append(q, k, v, (cl - 1).astype(np.int32), sl, oracle.rope_table(1e6, d_head, max_pos),
                              kc, vc)
    assert st == 0
    ref = oracle.paged_attention(q_ref, kc, vc, bt, cl, scale, nthreads=8)
    assert_attention_close(fused[3], ref, f"edge lengths d={d_head} G={Hq // Hkv}")


def test_step_bad_position_and_overlap(cuda_device):
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(3))
    B, Hq, Hkv, dh, nb = 3, 4, 2, 64, 8
    cl = np.array([5, 40, 0], np.int32)  # request 2 is empty: no append, a zero row
    bt = np.array([[0, -1, -1], [1, 2, 3], [-1, -1, -1]], np.int32)
    kc = bf16_normal(r, (nb, Hkv, 16, dh))
    vc = bf16_normal(r, (nb, Hkv, 16, dh))
    q, k, v = bf16_normal(r, (B, Hq, dh)), bf16_normal(r, (B, Hkv, dh)), bf16_normal(r, (B, Hkv, dh))
    max_pos = 16  # request 1 appends at position 39: past the table
    _, table = mi.mi_rope_table(1e6, dh, max_pos)
    d = mi.dims(B, Hq, Hkv, dh, nb, 3)
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=cuda_device)
    q_d = to_dev_u16(q, cuda_device)
    qo_d = torch.empty_like(q_d)
    out = torch.empty_like(q_d)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    args = (to_dev_u16(k, cuda_device), to_dev_u16(v, cuda_device), torch.from_numpy(table).to(cuda_device), max_pos,
            to_dev_i32(bt, cuda_device), to_dev_i32(cl, cuda_device), 0.125)
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)
    assert mi.mi_paged_decode_step(d, q_d, *args, qo_d, kc_d, vc_d, out, ws, dev_err=err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) & mi.MI_DEVERR_BAD_POS
    got = from_dev_u16(out)
    assert np.all(np.isfinite(oracle.bf16_to_f64(got)))
    assert np.all(got[2] == 0)
    # q_out over q (in place) is refused: other CTAs may still read q
    assert mi.mi_paged_decode_step(d, q_d, *args, q_d, kc_d, vc_d, out, ws, dev_err=err) == mi.MI_ERR_INVALID_ARG


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("name", ["qwen3_8b", "tiny", "qwen3_1p7b", "skewed", "empty_rows"])
def test_early_start_stack_matches_the_plain_stack(cuda_device, kv, name):
    """A stack of fused steps (every layer's own caches and q / k / v),
    called with MI_STEP_EARLY_START and two workspaces in turn, so that no
    step shares its workspace with the kernel just before it: every layer's
    q_out, cache and out carry the same bits as the stack called without the
    flag on one workspace, both eagerly and replayed from a CUDA graph
    (twice: a replay rewrites the same rows). Workloads: the Qwen3-8B
    serving layer at full size (persistent grid), the small ones (a grid
    cut to fewer CTAs than SMs) and the skewed batch, and the Qwen3-1.7B
    layer with two requests of length 0 (zero rows, nothing appended)."""
    import torch
    import bench
    mi = _mi()
    w = WORKLOADS["qwen3_1p7b" if name == "empty_rows" else name]
    L = 3
    fp8 = kv == "fp8"
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    if name == "empty_rows":
        cl = cl.copy()
        cl[[1, 5]] = 0
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    ks, vs = bench.fp8_scales(w)
    ks_d, vs_d = torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device)
    caches = []
    for layer in range(L):
        kc = torch.empty(shape, dtype=torch.uint8 if fp8 else torch.bfloat16, device=cuda_device)
        vc = torch.empty_like(kc)
        if fp8:
            bench.device_fill_fp8(w, layer, kc, vc, ks, vs)
        else:
            device_fill_cache(w, layer, kc, vc)
        caches.append((kc, vc))
    qkv = [tuple(to_dev_u16(a, cuda_device) for a in new_token_values(w, layer)) for layer in range(L)]
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    tab_d = torch.from_numpy(table).to(cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(cl, cuda_device)
    wsb = mi.mi_paged_decode_workspace_bytes(d) // 4 + 4
    ws = [torch.empty(wsb, dtype=torch.float32, device=cuda_device) for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)

    def run(cs, qo, out, flags):
        for layer in range(L):
            q_d, k_d, v_d = qkv[layer]
            kc, vc = cs[layer]
            wk = ws[layer % 2] if flags else ws[0]
            if fp8:
                st = mi.mi_paged_decode_step_fp8(d, q_d, k_d, v_d, tab_d, w.max_pos, bt_d, cl_d, ks_d, vs_d,
                                                 w.scale, qo[layer], kc, vc, out[layer], wk, dev_err=err,
                                                 flags=flags)
            else:
                st = mi.mi_paged_decode_step(d, q_d, k_d, v_d, tab_d, w.max_pos, bt_d, cl_d, w.scale, qo[layer], kc,
                                             vc, out[layer], wk, dev_err=err, flags=flags)
            assert st == 0, mi.status_string(st)

    def fresh():
        return ([(kc.clone(), vc.clone()) for kc, vc in caches],
                [torch.full_like(qkv[0][0], float("nan")) for _ in range(L)],
                [torch.full_like(qkv[0][0], float("nan")) for _ in range(L)])

    def same(a, b, what):
        ca, qa, oa = a
        cb, qb, ob = b
        for layer in range(L):
            assert torch.equal(qa[layer].view(torch.int16), qb[layer].view(torch.int16)), f"{what} q_out {layer}"
            assert torch.equal(oa[layer].view(torch.int16), ob[layer].view(torch.int16)), f"{what} out {layer}"
            for x, y in zip(ca[layer], cb[layer]):
                assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), f"{what} cache {layer}"

    plain = fresh()
    torch.cuda.synchronize()
    run(*plain, flags=0)
    torch.cuda.synchronize()
    for rep in range(2):   # the second pass finds its plans in the workspaces
        early = fresh()
        torch.cuda.synchronize()
        run(*early, flags=mi.MI_STEP_EARLY_START)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        same(plain, early, f"eager pass {rep}")
    graph_bufs = fresh()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(*graph_bufs, flags=mi.MI_STEP_EARLY_START)
    for rep in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        same(plain, graph_bufs, f"graph replay {rep}")
