"""GPU parity of the KV swap path: mi_kv_copy_blocks bit-exact against the
oracle's block copy (device to device, device to pinned host, pinned host to
device, block lists in device or pinned host memory), blocks not listed left
as they were; and a swap round trip on a serving batch (LRU victim out to a
pinned host cache, its blocks reused and overwritten, back into fresh blocks)
leaves every request's decode attention bitwise unchanged."""
import numpy as np
import pytest

from helpers import from_dev_u16, to_dev_i32, to_dev_u16
from oracle.pool import PoolModel
from oracle.swap import copy_blocks
from workloads import WORKLOADS, bf16_normal

pytestmark = pytest.mark.gpu

BS = 16


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


def _pinned_u16(a):
    import torch
    t = torch.empty(a.shape, dtype=torch.int16).pin_memory()
    t.numpy()[...] = a.view(np.int16)
    return t.view(torch.bfloat16)


@pytest.mark.parametrize("Hkv,d", [(2, 64), (8, 128)])
@pytest.mark.parametrize("route", ["d2d", "d2h", "h2d"])
def test_copy_blocks_bit_exact(cuda_device, Hkv, d, route):
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(Hkv * 7 + d))
    ns, nd = 40, 24
    sk, sv = bf16_normal(r, (ns, Hkv, BS, d)), bf16_normal(r, (ns, Hkv, BS, d))
    dk, dv = bf16_normal(r, (nd, Hkv, BS, d)), bf16_normal(r, (nd, Hkv, BS, d))
    si = r.choice(ns, size=17, replace=False).astype(np.int32)
    di = r.choice(nd, size=17, replace=False).astype(np.int32)
    on_host = {"d2d": (False, False), "d2h": (False, True), "h2d": (True, False)}[route]
    src = [(_pinned_u16(x) if on_host[0] else to_dev_u16(x, cuda_device)) for x in (sk, sv)]
    dst = [(_pinned_u16(x) if on_host[1] else to_dev_u16(x, cuda_device)) for x in (dk, dv)]
    # block lists: device for d2d, pinned host otherwise
    if route == "d2d":
        si_t, di_t = to_dev_i32(si, cuda_device), to_dev_i32(di, cuda_device)
    else:
        si_t, di_t = torch.from_numpy(si).pin_memory(), torch.from_numpy(di).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dims = mi.dims(1, Hkv, Hkv, d, 1, 1)
    assert mi.mi_kv_copy_blocks(dims, src[0], src[1], ns, si_t, dst[0], dst[1], nd, di_t, len(si), err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    copy_blocks(sk, si, dk, di)
    copy_blocks(sv, si, dv, di)
    assert np.array_equal(from_dev_u16(dst[0]), dk)
    assert np.array_equal(from_dev_u16(dst[1]), dv)


def test_copy_blocks_bad_id_and_pageable_memory(cuda_device):
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(5))
    k = to_dev_u16(bf16_normal(r, (8, 2, BS, 64)), cuda_device)
    v = to_dev_u16(bf16_normal(r, (8, 2, BS, 64)), cuda_device)
    hk, hv = torch.empty_like(k, device="cpu").pin_memory(), torch.empty_like(v, device="cpu").pin_memory()
    before = from_dev_u16(hk).copy()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dims = mi.dims(1, 2, 2, 64, 1, 1)
    si, di = to_dev_i32(np.array([1, 9], np.int32), cuda_device), to_dev_i32(np.array([0, 1], np.int32), cuda_device)
    assert mi.mi_kv_copy_blocks(dims, k, v, 8, si, hk, hv, 8, di, 2, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) & mi.MI_DEVERR_BAD_BLOCK
    got = from_dev_u16(hk)
    assert np.array_equal(got[0], from_dev_u16(k)[1]) and np.array_equal(got[1], before[1])
    pageable = torch.empty_like(k, device="cpu")
    assert mi.mi_kv_copy_blocks(dims, k, v, 8, si, pageable, hv, 8, di, 1, err) == mi.MI_ERR_INVALID_ARG


def test_swap_round_trip_keeps_decode_attention_bitwise(cuda_device):
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_1p7b"]
    r = np.random.Generator(np.random.PCG64(8))
    nb = w.num_blocks
    dev, model = mi.Pool(nb, 64, w.max_blocks_per_seq), PoolModel(nb, 64, w.max_blocks_per_seq)
    host = mi.Pool(512, 64, w.max_blocks_per_seq)
    lens = r.integers(200, 1500, size=w.B)
    for b in range(w.B):
        assert dev.alloc(b, int(lens[b])) == 0 and model.alloc(b, int(lens[b])) == 0
    assert dev.touch([0, 2, 4, 6]) == 0 and model.touch([0, 2, 4, 6]) == 0
    kc = to_dev_u16(bf16_normal(r, (nb, w.Hkv, BS, w.head_dim)), cuda_device)
    vc = to_dev_u16(bf16_normal(r, (nb, w.Hkv, BS, w.head_dim)), cuda_device)
    q = to_dev_u16(bf16_normal(r, (w.B, w.Hq, w.head_dim)), cuda_device)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, nb, w.max_blocks_per_seq)
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)

    def attend():
        bt, cl, _ = dev.batch_meta(list(range(w.B)))
        out = torch.empty_like(q)
        assert mi.mi_paged_decode_attention(d, q, kc, vc, to_dev_i32(bt, cuda_device), to_dev_i32(cl, cuda_device),
                                            w.scale, out, ws, dev_err=err) == 0
        torch.cuda.synchronize()
        return from_dev_u16(out)

    before = attend()
    victim = dev.lru_victim()
    assert victim == model.lru_victim() == 1   # untouched since its alloc, the oldest of 1, 3, 5, 7
    st, blocks = dev.swap_out(victim)
    assert (st, blocks) == model.swap_out(victim)
    assert host.alloc(victim, int(lens[victim])) == 0
    hb = mi.mi_kv_pool_seq_blocks(host.handle, victim)
    hk = torch.empty((512, w.Hkv, BS, w.head_dim), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    side = torch.cuda.Stream(cuda_device)
    dims = mi.dims(1, w.Hkv, w.Hkv, w.head_dim, 1, 1)
    src_ids, dst_ids = to_dev_i32(blocks, cuda_device), to_dev_i32(hb, cuda_device)  # held until synced
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    assert mi.mi_kv_copy_blocks(dims, kc, vc, nb, src_ids, hk, hv, 512, dst_ids, len(blocks), err, side) == 0
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    # a new sequence takes the freed blocks and fills them with NaN bits
    assert dev.alloc(40, len(blocks) * BS) == 0
    taken = mi.mi_kv_pool_seq_blocks(dev.handle, 40)
    assert set(int(x) for x in taken) == set(blocks)
    idx = torch.from_numpy(taken.astype(np.int64)).to(cuda_device)
    kc.view(torch.int16)[idx] = 0x7FA5
    vc.view(torch.int16)[idx] = 0x7FA5
    assert dev.free(40) == 0
    # make room elsewhere so the victim comes back to other blocks
    assert dev.alloc(41, 64 * BS) == 0
    st, new = dev.swap_in(victim)
    assert st == 0 and len(new) == len(blocks) and set(new) != set(blocks)
    src2, dst2 = to_dev_i32(hb, cuda_device), to_dev_i32(np.array(new, np.int32), cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    assert mi.mi_kv_copy_blocks(dims, hk, hv, 512, src2, kc, vc, nb, dst2, len(new), err, side) == 0
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    after = attend()
    del src_ids, dst_ids, src2, dst2
    assert int(err.item()) == 0
    assert np.array_equal(before, after)
