"""GPU parity of the FP8 (e4m3, per-KV-head scale) KV path against the
oracle: mi_paged_kv_append_fp8 bit-exact (q_out and both caches, every other
byte untouched, saturation and subnormal codes included), and
mi_paged_decode_attention_fp8 within the attention tolerance of the fp64
oracle over the dequantised caches, on the small workloads in full and on a
full-size serving layer by sampled requests; paging invariance bitwise, edge
lengths, and the bad-scale error bit."""
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


def test_fp8_full_size_serving_layer_sampled(cuda_device):
    """Qwen3-8B-shaped layer at full size (e4m3 caches filled on the device),
    persistent grid; the oracle recomputes 12 requests."""
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_8b"]
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    ks, vs = _scales(w.Hkv, w.seed)
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    g = torch.Generator(device=cuda_device)
    g.manual_seed(w.seed)
    caches = []
    for sc in (ks, vs):
        x = torch.randn(shape, generator=g, device=cuda_device) / torch.from_numpy(sc).to(cuda_device)[None, :, None, None]
        caches.append(x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))  # torch casts overflow to NaN
        del x
    kc_d, vc_d = caches
    q, _, _ = new_token_values(w, 0)
    q_d = to_dev_u16(q, cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    out, err = _attend(mi, d, q_d, kc_d, vc_d, torch.from_numpy(ks).to(cuda_device),
                       torch.from_numpy(vs).to(cuda_device), bt, cl, w.scale, cuda_device)
    assert err == 0
    order = np.argsort(cl)
    sample = sorted(set(order[:4].tolist() + order[-4:].tolist() + [5, 17, 33, 50]))
    used = sorted({int(x) for b in sample for x in bt[b, :-(-int(cl[b]) // BLOCK)]})
    remap = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.int64, device=cuda_device)
    kc_s, vc_s = kc_d[idx].cpu().numpy(), vc_d[idx].cpu().numpy()
    bt_s = np.full((len(sample), bt.shape[1]), -1, np.int32)
    for i, b in enumerate(sample):
        n = -(-int(cl[b]) // BLOCK)
        bt_s[i, :n] = [remap[int(x)] for x in bt[b, :n]]
    ref = oracle.paged_attention_fp8(q[sample], kc_s, vc_s, ks, vs, bt_s, cl[sample], w.scale, nthreads=8)
    assert_attention_close(out[sample], ref, "fp8 qwen3_8b sampled")


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
