"""GPU parity of the FP8 (e4m3, per-KV-head scale) KV path against the
oracle: mi_paged_kv_append_fp8 bit-exact (q_out and both caches, every other
byte untouched, saturation and subnormal codes included), and
mi_paged_decode_attention_fp8 within the attention tolerance of the fp64
oracle over the dequantised caches, on the small workloads in full and on a
full-size serving layer (every request and head); paging invariance bitwise,
edge lengths, and the bad-scale error bit. The fused FP8 decode step
(mi_paged_decode_step_fp8) writes what the FP8 append writes, bit for bit,
and its output is within the tolerance of the FP8 attention's and the
oracle's."""
import numpy as np
import pytest

import oracle
from helpers import assert_attention_close, from_dev_u16, grow, pools_for, to_dev_i32, to_dev_u16
from workloads import BLOCK, WORKLOADS, bf16_normal, history_cache, new_token_values

pytestmark = pytest.mark.gpu


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


def _scales(Hkv, seed):
    """Per-head scales spanning about 3..6 standard deviations at e4m3's 448."""
    r = np.random.Generator(np.random.PCG64(seed))
    ks = ((3.0 + 3.0 * r.random(Hkv)) / 448.0).astype(np.float32)
    vs = ((3.0 + 3.0 * r.random(Hkv)) / 448.0).astype(np.float32)
    return ks, vs


def _quantise(c16, scale):
    """bf16 cache -> e4m3 codes with the oracle's rule (fp32 quotient, then
    e4m3); NaN canaries stay NaN codes."""
    x = oracle.bf16_to_f64(c16).astype(np.float32) / scale[None, :, None, None]
    return oracle.e4m3_from_f64(x.astype(np.float64))


def _to_dev_u8(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(device)


def _workspace(mi, d, device):
    import torch
    n = mi.mi_paged_decode_workspace_bytes(d)
    assert n > 0
    return torch.empty(n // 4 + 4, dtype=torch.float32, device=device)


def _attend(mi, d, q_d, kc_d, vc_d, ks_d, vs_d, bt, cl, scale, device):
    import torch
    out = torch.full(q_d.shape, float("nan"), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    st = mi.mi_paged_decode_attention_fp8(d, q_d, kc_d, vc_d, ks_d, vs_d, to_dev_i32(bt, device),
                                          to_dev_i32(cl, device), scale, out, _workspace(mi, d, device),
                                          dev_err=err)
    assert st == 0, mi.status_string(st)
    torch.cuda.synchronize()
    return from_dev_u16(out), int(err.item())


def _small_case(name, device):
    """FP8 history plus one token appended through the library; the oracle
    appends the same token to its own copies."""
    import torch
    mi = _mi()
    w = WORKLOADS[name]
    lib, model, ctx = pools_for(w)
    bt_hist, _, _ = lib.batch_meta(range(w.B))
    grow(lib, w.B, ctx + 1)
    grow(model, w.B, ctx + 1)
    bt, cl, sl = lib.batch_meta(range(w.B))
    ks, vs = _scales(w.Hkv, w.seed)
    kc16, vc16 = history_cache(w, 0, bt_hist, ctx)
    kc8, vc8 = _quantise(kc16, ks), _quantise(vc16, vs)
    q, k, v = new_token_values(w, 0)
    pos = (cl - 1).astype(np.int32)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    kc_d, vc_d = _to_dev_u8(kc8, device), _to_dev_u8(vc8, device)
    ks_d, vs_d = torch.from_numpy(ks).to(device), torch.from_numpy(vs).to(device)
    q_d = to_dev_u16(q, device)
    qo_d = torch.empty_like(q_d)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    assert mi.mi_paged_kv_append_fp8(d, q_d, to_dev_u16(k, device), to_dev_u16(v, device), to_dev_i32(pos, device),
                                     to_dev_i32(sl, device), torch.from_numpy(table).to(device), w.max_pos, qo_d,
                                     kc_d, vc_d, ks_d, vs_d, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q_ref, st = oracle.append_fp8(q, k, v, pos, model.batch_meta(range(w.B))[2],
                                  oracle.rope_table(w.theta, w.head_dim, w.max_pos), ks, vs, kc8, vc8)
    assert st == 0
    return w, d, q_ref, kc8, vc8, ks, vs, bt, cl, qo_d, kc_d, vc_d, ks_d, vs_d


@pytest.mark.parametrize("name", ["tiny", "qwen3_1p7b", "skewed"])
def test_fp8_append_bit_exact_and_attention_matches_oracle(cuda_device, name):
    mi = _mi()
    w, d, q, kc8, vc8, ks, vs, bt, cl, q_d, kc_d, vc_d, ks_d, vs_d = _small_case(name, cuda_device)
    assert np.array_equal(from_dev_u16(q_d), q)
    assert np.array_equal(kc_d.cpu().numpy(), kc8)
    assert np.array_equal(vc_d.cpu().numpy(), vc8)
    ref = oracle.paged_attention_fp8(q, kc8, vc8, ks, vs, bt, cl, w.scale, nthreads=8)
    out, err = _attend(mi, d, q_d, kc_d, vc_d, ks_d, vs_d, bt, cl, w.scale, cuda_device)
    assert err == 0
    assert_attention_close(out, ref, f"fp8 {name}")


def test_fp8_append_extreme_values(cuda_device):
    """Saturation past 448 * scale, e4m3 subnormals, zeros of both signs and
    ties, through the library append and the oracle's."""
    import torch
    mi = _mi()
    B, Hq, Hkv, dh, nb = 4, 4, 2, 64, 8
    r = np.random.Generator(np.random.PCG64(9))
    ks = np.array([0.01, 2.0], np.float32)
    vs = np.array([0.5, 0.001], np.float32)
    special = np.array([1e30, -1e30, 5.0, -5.0, 4.48, 4.6, 1e-6, -1e-6, 0.0, -0.0, 2.0 ** -12, 3e-5,
                        0.0234375, 1.1875, 300.0, -0.4, 0.005, -0.001], np.float64)
    k = r.choice(special, size=(B, Hkv, dh)) * r.choice([1.0, 0.5, 3.0], size=(B, Hkv, dh))
    v = r.choice(special, size=(B, Hkv, dh))
    k16, v16 = oracle.f64_to_bf16(k), oracle.f64_to_bf16(v)
    q16 = bf16_normal(r, (B, Hq, dh))
    pos = np.array([0, 3, 16, 40], np.int32)
    slots = np.array([1, 17, 40, 127], np.int32)
    table = oracle.rope_table(1e6, dh, 64)
    kc8 = r.integers(0, 256, size=(nb, Hkv, BLOCK, dh), dtype=np.uint8)
    vc8 = r.integers(0, 256, size=(nb, Hkv, BLOCK, dh), dtype=np.uint8)
    d = mi.dims(B, Hq, Hkv, dh, nb, 4)
    kc_d, vc_d = _to_dev_u8(kc8, cuda_device), _to_dev_u8(vc8, cuda_device)
    qo_d = torch.empty((B, Hq, dh), dtype=torch.bfloat16, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    assert mi.mi_paged_kv_append_fp8(d, to_dev_u16(q16, cuda_device), to_dev_u16(k16, cuda_device),
                                     to_dev_u16(v16, cuda_device), to_dev_i32(pos, cuda_device),
                                     to_dev_i32(slots, cuda_device), torch.from_numpy(table).to(cuda_device), 64,
                                     qo_d, kc_d, vc_d, torch.from_numpy(ks).to(cuda_device),
                                     torch.from_numpy(vs).to(cuda_device), err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q_ref, st = oracle.append_fp8(q16, k16, v16, pos, slots, table, ks, vs, kc8, vc8)
    assert st == 0
    assert np.array_equal(from_dev_u16(qo_d), q_ref)
    assert np.array_equal(kc_d.cpu().numpy(), kc8)
    assert np.array_equal(vc_d.cpu().numpy(), vc8)
    rows_k = kc8[slots // BLOCK, :, slots % BLOCK]
    rows_v = vc8[slots // BLOCK, :, slots % BLOCK]
    assert (rows_k == 0x7E).any() and (rows_k == 0xFE).any()          # saturated both ways
    sub = rows_v[:, 0] & 0x7F                                          # head 0: v / 0.5
    assert ((sub > 0) & (sub < 8)).any()                               # e4m3 subnormal codes


def test_fp8_bad_scale_skips_the_head(cuda_device):
    import torch
    mi = _mi()
    B, Hq, Hkv, dh, nb = 2, 4, 2, 64, 4
    r = np.random.Generator(np.random.PCG64(10))
    q16, k16, v16 = (bf16_normal(r, (B, H, dh)) for H in (Hq, Hkv, Hkv))
    kc_d = torch.zeros((nb, Hkv, BLOCK, dh), dtype=torch.uint8, device=cuda_device)
    vc_d = torch.zeros_like(kc_d)
    ks = torch.tensor([0.0, 0.02], device=cuda_device)
    vs = torch.tensor([0.02, float("inf")], device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    d = mi.dims(B, Hq, Hkv, dh, nb, 2)
    table = torch.from_numpy(oracle.rope_table(1e6, dh, 8)).to(cuda_device)
    q_d = to_dev_u16(q16, cuda_device)
    assert mi.mi_paged_kv_append_fp8(d, q_d, to_dev_u16(k16, cuda_device), to_dev_u16(v16, cuda_device),
                                     to_dev_i32(np.array([0, 1], np.int32), cuda_device),
                                     to_dev_i32(np.array([0, 20], np.int32), cuda_device), table, 8, q_d,
                                     kc_d, vc_d, ks, vs, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) & mi.MI_DEVERR_BAD_SCALE
    kc, vc = kc_d.cpu().numpy(), vc_d.cpu().numpy()
    assert not kc[:, 0].any() and kc[:, 1].any()                  # head 0 of K skipped
    assert vc[:, 0].any() and not vc[:, 1].any()                  # head 1 of V skipped


def test_fp8_full_size_serving_layer(cuda_device):
    """Qwen3-8B-shaped layer at full size (e4m3 caches filled on the device),
    persistent grid: every request and head against the oracle over the
    blocks the requests use (copied back and renumbered)."""
    import os
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_8b"]
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    ks, vs = _scales(w.Hkv, w.seed)
    kc_d, vc_d = _device_fp8_caches(w, ks, vs, cuda_device)
    q, _, _ = new_token_values(w, 0)
    q_d = to_dev_u16(q, cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    out, err = _attend(mi, d, q_d, kc_d, vc_d, torch.from_numpy(ks).to(cuda_device),
                       torch.from_numpy(vs).to(cuda_device), bt, cl, w.scale, cuda_device)
    assert err == 0
    kc_s, vc_s, bt_s = _used_blocks_u8(kc_d, vc_d, bt, cl)
    ref = oracle.paged_attention_fp8(q, kc_s, vc_s, ks, vs, bt_s, cl, w.scale, nthreads=os.cpu_count() or 8)
    assert_attention_close(out, ref, "fp8 qwen3_8b")


def _device_fp8_caches(w, ks, vs, device):
    """e4m3 caches [num_blocks][Hkv][16][d] of N(0,1) / scale, clamped to
    +-448 (torch casts overflow to NaN), from a seeded device generator."""
    import torch
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    caches = []
    for sc in (ks, vs):
        x = torch.randn(shape, generator=g, device=device) / torch.from_numpy(sc).to(device)[None, :, None, None]
        caches.append(x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))
        del x
    return caches


def _used_blocks_u8(kc_d, vc_d, bt, cl):
    """Host copies of the blocks the requests use, renumbered, and the
    tables rewritten to the new numbers (data movement only)."""
    import torch
    live = [bt[b, :-(-max(int(cl[b]), 0) // BLOCK)] for b in range(len(cl))]
    used = sorted({int(x) for row in live for x in row})
    remap = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.int64, device=kc_d.device)
    bt_s = np.full(bt.shape, -1, np.int32)
    for i, row in enumerate(live):
        bt_s[i, :len(row)] = [remap[int(x)] for x in row]
    return kc_d[idx].cpu().numpy(), vc_d[idx].cpu().numpy(), bt_s


def _fp8_both(device, d, q, k, v, table, max_pos, bt, cl, kc8, vc8, ks, vs, scale):
    """(two-call results, fused-step results), each (q_out, k_cache, v_cache,
    out, err), on fresh device copies of the same e4m3 caches."""
    import torch
    mi = _mi()
    ws = _workspace(mi, d, device)
    tab_d = torch.from_numpy(table).to(device)
    bt_d, cl_d = to_dev_i32(bt, device), to_dev_i32(cl, device)
    ks_d, vs_d = torch.from_numpy(ks).to(device), torch.from_numpy(vs).to(device)
    pos = (cl - 1).astype(np.int32)
    sl = np.array([bt[b, (cl[b] - 1) // 16] * 16 + (cl[b] - 1) % 16 if cl[b] > 0 else -1 for b in range(len(cl))],
                  np.int32)
    res = []
    for fused in (False, True):
        q_d, k_d, v_d = to_dev_u16(q, device), to_dev_u16(k, device), to_dev_u16(v, device)
        kc_d, vc_d = _to_dev_u8(kc8, device), _to_dev_u8(vc8, device)
        qo_d = torch.full_like(q_d, float("nan"))
        out = torch.full_like(q_d, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=device)
        if fused:
            st = mi.mi_paged_decode_step_fp8(d, q_d, k_d, v_d, tab_d, max_pos, bt_d, cl_d, ks_d, vs_d, scale, qo_d,
                                             kc_d, vc_d, out, ws, dev_err=err)
            assert st == 0, mi.status_string(st)
        else:
            live = cl > 0
            if live.any():
                rows = np.flatnonzero(live)
                d_app = mi.dims(len(rows), d.Hq, d.Hkv, d.head_dim, d.num_blocks, d.max_blocks_per_seq)
                qa, ka, va = (to_dev_u16(a[rows], device) for a in (q, k, v))
                qoa = torch.empty_like(qa)
                assert mi.mi_paged_kv_append_fp8(d_app, qa, ka, va, to_dev_i32(pos[rows], device),
                                                 to_dev_i32(sl[rows], device), tab_d, max_pos, qoa, kc_d, vc_d,
                                                 ks_d, vs_d, err) == 0
                qo_d[torch.from_numpy(rows).to(device)] = qoa
            assert mi.mi_paged_decode_attention_fp8(d, qo_d, kc_d, vc_d, ks_d, vs_d, bt_d, cl_d, scale, out, ws,
                                                    dev_err=err) == 0
        torch.cuda.synchronize()
        res.append((from_dev_u16(qo_d), kc_d.cpu().numpy(), vc_d.cpu().numpy(), from_dev_u16(out), int(err.item())))
    return res


@pytest.mark.parametrize("name", ["tiny", "qwen3_1p7b", "skewed"])
def test_fp8_step_matches_two_calls_and_oracle(cuda_device, name):
    """mi_paged_decode_step_fp8 (RoPE, quantised cache row and e4m3 attention
    in one launch) gives q_out and both caches bit for bit as the FP8 append,
    the output within the tolerance of the FP8 attention after it (another
    grid, another split), and the oracle's own FP8 append + attention within
    the tolerance."""
    mi = _mi()
    w = WORKLOADS[name]
    lib, model, ctx = pools_for(w)
    bt_hist, _, _ = lib.batch_meta(range(w.B))
    grow(lib, w.B, ctx + 1)
    grow(model, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    ks, vs = _scales(w.Hkv, w.seed)
    kc16, vc16 = history_cache(w, 0, bt_hist, ctx)
    kc8, vc8 = _quantise(kc16, ks), _quantise(vc16, vs)
    q, k, v = new_token_values(w, 0)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    two, fused = _fp8_both(cuda_device, d, q, k, v, table, w.max_pos, bt, cl, kc8, vc8, ks, vs, w.scale)
    for i, what in enumerate(("q_out", "k_cache", "v_cache")):
        assert np.array_equal(two[i], fused[i]), f"{what} differs from the two FP8 calls"
    # the fused e4m3 step runs two CTAs per SM, the e4m3 attention three: a
    # different split, so the outputs agree to the attention's rounding
    assert_attention_close(fused[3], oracle.bf16_to_f64(two[3]), f"fp8 fused step vs two calls {name}")
    assert two[4] == fused[4] == 0
    pos = (cl - 1).astype(np.int32)
    q_ref, st = oracle.append_fp8(q, k, v, pos, model.batch_meta(range(w.B))[2],
                                  oracle.rope_table(w.theta, w.head_dim, w.max_pos), ks, vs, kc8, vc8)
    assert st == 0
    assert np.array_equal(fused[0], q_ref)
    assert np.array_equal(fused[1], kc8) and np.array_equal(fused[2], vc8)
    ref = oracle.paged_attention_fp8(q_ref, kc8, vc8, ks, vs, bt, cl, w.scale, nthreads=8)
    assert_attention_close(fused[3], ref, f"fp8 fused step {name}")


@pytest.mark.parametrize("d_head,Hq,Hkv", [(128, 8, 2), (64, 4, 2), (128, 7, 1), (64, 8, 8)])
def test_fp8_step_edge_lengths(cuda_device, d_head, Hq, Hkv):
    """Contexts of 0, 1, 15, 16, 17, 31, 32, 33 and 200 tokens after the
    append (the new token first, last or alone in its block), NaN codes in
    every unused cache row: the fused FP8 step writes the same q_out and cache
    rows as the two FP8 calls, and its output is within the tolerance of
    theirs and of the oracle's; the empty request gets a zero row."""
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(d_head * 7 + Hq))
    cl = np.array([1, 15, 16, 17, 0, 31, 32, 33, 200], np.int32)
    B = len(cl)
    nblk = -(-np.maximum(cl, 0) // 16)
    nb = int(nblk.sum()) + 5
    mbps = int(nblk.max())
    perm = r.permutation(nb)
    bt = np.full((B, mbps), -1, np.int32)
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    ks, vs = _scales(Hkv, 5)
    kc8 = np.full((nb, Hkv, 16, d_head), 0x7F, np.uint8)
    vc8 = np.full((nb, Hkv, 16, d_head), 0xFF, np.uint8)
    for b in range(B):
        for t in range(cl[b] - 1):  # history; the step writes row cl - 1
            kc8[bt[b, t // 16], :, t % 16] = _quantise(bf16_normal(r, (1, Hkv, 1, d_head)), ks)[0, :, 0]
            vc8[bt[b, t // 16], :, t % 16] = _quantise(bf16_normal(r, (1, Hkv, 1, d_head)), vs)[0, :, 0]
    q, k, v = bf16_normal(r, (B, Hq, d_head)), bf16_normal(r, (B, Hkv, d_head)), bf16_normal(r, (B, Hkv, d_head))
    max_pos = 256
    _, table = mi.mi_rope_table(1e6, d_head, max_pos)
    d = mi.dims(B, Hq, Hkv, d_head, nb, mbps)
    scale = 1.0 / np.sqrt(d_head)
    two, fused = _fp8_both(cuda_device, d, q, k, v, table, max_pos, bt, cl, kc8, vc8, ks, vs, scale)
    for i, what in enumerate(("q_out", "k_cache", "v_cache")):
        assert np.array_equal(two[i], fused[i]), f"{what} differs from the two FP8 calls"
    assert_attention_close(fused[3], oracle.bf16_to_f64(two[3]), "fp8 fused step vs two calls, edges")
    assert np.all(fused[3][cl == 0] == 0)
    live = cl > 0
    pos = (cl - 1).astype(np.int32)
    sl = np.array([bt[b, pos[b] // 16] * 16 + pos[b] % 16 for b in np.flatnonzero(live)], np.int32)
    kc_h, vc_h = kc8.copy(), vc8.copy()
    q_ref, st = oracle.append_fp8(q[live], k[live], v[live], pos[live], sl, oracle.rope_table(1e6, d_head, max_pos),
                                  ks, vs, kc_h, vc_h)
    assert st == 0
    assert np.array_equal(fused[0][live], q_ref)
    assert np.array_equal(fused[1], kc_h) and np.array_equal(fused[2], vc_h)
    qa = fused[0].copy()
    ref = oracle.paged_attention_fp8(qa, kc_h, vc_h, ks, vs, bt, cl, scale, nthreads=8)
    assert_attention_close(fused[3], ref, f"fp8 step edges d={d_head} G={Hq // Hkv}")


def test_fp8_step_bad_scale_skips_the_row(cuda_device):
    """A KV head whose K (or V) scale is not a positive finite number: the
    fused FP8 step, like the FP8 append, sets MI_DEVERR_BAD_SCALE and leaves
    that head's K (or V) cache row as it was."""
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(21))
    B, Hq, Hkv, dh = 3, 4, 2, 64
    cl = np.array([5, 20, 33], np.int32)
    nb = 8
    bt = np.array([[0, -1, -1], [1, 2, -1], [3, 4, 5]], np.int32)
    ks = np.array([0.0, 0.02], np.float32)
    vs = np.array([0.02, np.inf], np.float32)
    kc8 = r.integers(0, 0x70, size=(nb, Hkv, 16, dh), dtype=np.uint8)
    vc8 = r.integers(0, 0x70, size=(nb, Hkv, 16, dh), dtype=np.uint8)
    q, k, v = bf16_normal(r, (B, Hq, dh)), bf16_normal(r, (B, Hkv, dh)), bf16_normal(r, (B, Hkv, dh))
    _, table = mi.mi_rope_table(1e6, dh, 64)
    d = mi.dims(B, Hq, Hkv, dh, nb, 3)
    two, fused = _fp8_both(cuda_device, d, q, k, v, table, 64, bt, cl, kc8, vc8, ks, vs, 0.125)
    assert fused[4] & mi.MI_DEVERR_BAD_SCALE and two[4] & mi.MI_DEVERR_BAD_SCALE
    for i, what in enumerate(("q_out", "k_cache", "v_cache")):
        assert np.array_equal(two[i], fused[i]), what
    for b in range(B):
        blk, off = bt[b, (cl[b] - 1) // 16], (cl[b] - 1) % 16
        assert np.array_equal(fused[1][blk, 0, off], kc8[blk, 0, off])      # K of head 0: not written
        assert not np.array_equal(fused[1][blk, 1, off], kc8[blk, 1, off])  # K of head 1: written
        assert np.array_equal(fused[2][blk, 1, off], vc8[blk, 1, off])      # V of head 1: not written


@pytest.mark.parametrize("d_head,Hq,Hkv", [(64, 8, 2), (128, 16, 2), (128, 32, 8), (64, 7, 7)])
def test_fp8_edge_lengths_and_paging_invariance(cuda_device, d_head, Hq, Hkv):
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(d_head + Hq))
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 200, 0, 1000], np.int32)
    B = len(lens)
    nblk = [-(-int(n) // BLOCK) for n in lens]
    nb = sum(nblk) + 5
    mbps = max(nblk)
    ks, vs = _scales(Hkv, 3)
    kc8 = _quantise(bf16_normal(r, (nb, Hkv, BLOCK, d_head)), ks)
    vc8 = _quantise(bf16_normal(r, (nb, Hkv, BLOCK, d_head)), vs)
    perm = r.permutation(nb)
    bt = np.full((B, mbps), -1, np.int32)
    i = 0
    for b in range(B):
        for j in range(nblk[b]):
            bt[b, j] = perm[i]; i += 1
        tail = int(lens[b]) % BLOCK
        if tail:  # NaN codes past the context in the last block
            kc8[bt[b, nblk[b] - 1], :, tail:] = 0x7F
            vc8[bt[b, nblk[b] - 1], :, tail:] = 0xFF
    q = bf16_normal(r, (B, Hq, d_head))
    d = mi.dims(B, Hq, Hkv, d_head, nb, mbps)
    ks_d, vs_d = torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device)
    q_d = to_dev_u16(q, cuda_device)
    out, err = _attend(mi, d, q_d, _to_dev_u8(kc8, cuda_device), _to_dev_u8(vc8, cuda_device), ks_d, vs_d, bt,
                       lens, 0.1, cuda_device)
    assert err == 0
    ref = oracle.paged_attention_fp8(q, kc8, vc8, ks, vs, bt, lens, 0.1, nthreads=8)
    assert_attention_close(out, ref, f"fp8 edges d={d_head} G={Hq // Hkv}")
    assert np.all(out[lens == 0] == 0)
    # the same caches with every block moved: bitwise the same output
    p2 = r.permutation(nb)
    kc2, vc2 = np.empty_like(kc8), np.empty_like(vc8)
    kc2[p2], vc2[p2] = kc8, vc8
    bt2 = np.where(bt >= 0, p2[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, _ = _attend(mi, d, q_d, _to_dev_u8(kc2, cuda_device), _to_dev_u8(vc2, cuda_device), ks_d, vs_d, bt2,
                      lens, 0.1, cuda_device)
    assert np.array_equal(out, out2)
