"""GPU parity of mi_kv_copy_rows and of a KV swap over INT8 caches.

* mi_kv_copy_rows copies rows of 8 B (group maxima of two KV heads, 4-byte
  words), 32 B, 16 KB (an INT8 block of 8 heads at d = 128) and 128 KB (a
  sequence's open-group rows) bit for bit against numpy indexing (the
  oracle's block copy), device to device, device to pinned host and back;
  rows not listed are left as they were; a bad id is flagged and skipped.
* A swap round trip of one sequence of an INT8 batch: its blocks' codes, its
  blocks' group maxima and its open-group rows go to pinned host memory, the
  device copies are overwritten, and everything comes back into other blocks
  and another slot. The next decode step (INT8 append + INT8 attention) then
  gives bit for bit what it gives on the state that never moved."""
import numpy as np
import pytest

import oracle
from helpers import from_dev_u16, to_dev_i32, to_dev_u16
from oracle.swap import copy_blocks
from workloads import bf16_normal

pytestmark = pytest.mark.gpu

BS = 16


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


@pytest.mark.parametrize("row_bytes", [8, 32, 16384, 131072])
@pytest.mark.parametrize("route", ["d2d", "d2h", "h2d"])
def test_copy_rows_bit_exact(cuda_device, row_bytes, route):
    import torch
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(row_bytes + len(route)))
    ns, nd, n = 40, 50, 17
    src = r.integers(0, 256, size=(ns, row_bytes), dtype=np.uint8)
    dst = r.integers(0, 256, size=(nd, row_bytes), dtype=np.uint8)
    si = r.choice(ns, n, replace=False).astype(np.int32)
    di = r.choice(nd, n, replace=False).astype(np.int32)
    want = dst.copy()
    copy_blocks(src, si, want, di)

    def place(a, host):
        t = torch.from_numpy(a.copy())
        return t.pin_memory() if host else t.to(cuda_device)
    s_t = place(src, route == "h2d")
    d_t = place(dst, route == "d2h")
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    assert mi.mi_kv_copy_rows(s_t, ns, to_dev_i32(si, cuda_device), d_t, nd, to_dev_i32(di, cuda_device), n,
                              row_bytes, err) == mi.MI_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(d_t.cpu().numpy(), want)


def test_copy_rows_bad_id_and_arguments(cuda_device):
    import torch
    mi = _mi()
    src = torch.arange(64, dtype=torch.int32, device=cuda_device).view(16, 4)
    dst = torch.full((8, 4), -1, dtype=torch.int32, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    si, di = to_dev_i32(np.array([3, 99, 5], np.int32), cuda_device), to_dev_i32(np.array([0, 1, 2], np.int32),
                                                                                 cuda_device)
    assert mi.mi_kv_copy_rows(src, 16, si, dst, 8, di, 3, 16, err) == mi.MI_OK
    torch.cuda.synchronize()
    assert int(err.item()) & mi.MI_DEVERR_BAD_BLOCK
    got = dst.cpu().numpy()
    assert got[0].tolist() == [12, 13, 14, 15] and (got[1] == -1).all() and got[2].tolist() == [20, 21, 22, 23]
    assert mi.mi_kv_copy_rows(src, 16, si, dst, 8, di, 3, 6, err) == mi.MI_ERR_INVALID_ARG    # not a multiple of 4
    pageable = torch.zeros((8, 4), dtype=torch.int32)
    assert mi.mi_kv_copy_rows(src, 16, si, pageable, 8, di, 3, 16, err) == mi.MI_ERR_INVALID_ARG


def _int8_batch(seed, lens, Hq=8, Hkv=2, d=128, spare=80):
    r = np.random.Generator(np.random.PCG64(seed))
    B = len(lens)
    nblk = [-(-(n + 1) // BS) for n in lens]          # room for the appended token
    nb = sum(nblk) + spare
    perm = r.permutation(nb)
    bt = np.full((B, max(nblk) + 1), -1, np.int32)
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    kc = bf16_normal(r, (nb, Hkv, BS, d))
    vc = bf16_normal(r, (nb, Hkv, BS, d))
    slots = np.arange(B, dtype=np.int32)
    st = oracle.int8_state(nb, Hkv, d, B + 2)
    assert oracle.int8_from_bf16_cache(kc, vc, bt, np.array(lens, np.int32), slots, st) == 0
    q, k, v = (bf16_normal(r, (B, H, d)) for H in (Hq, Hkv, Hkv))
    free = perm[i:]                                     # blocks nobody holds
    return r, st, bt, slots, q, k, v, free


def _step(mi, device, st, bt, cl, slots, q, k, v, Hq, table):
    """One INT8 append + attention on device copies of `st`; returns
    (q_out bits, out bits, state on the host)."""
    import torch
    nb, Hkv = st["k_amax"].shape
    d = st["k8"].shape[-1]
    B = q.shape[0]
    k8, v8 = torch.from_numpy(st["k8"]).to(device), torch.from_numpy(st["v8"]).to(device)
    ka = torch.from_numpy(st["k_amax"].ravel().copy()).to(device)
    va = torch.from_numpy(st["v_amax"].ravel().copy()).to(device)
    ko, vo = to_dev_u16(st["k_open"], device), to_dev_u16(st["v_open"], device)
    dims = mi.dims(B, Hq, Hkv, d, nb, bt.shape[1])
    qo = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=device)
    out = torch.empty_like(qo)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    bt_d, cl_d = to_dev_i32(bt, device), to_dev_i32(cl, device)
    assert mi.mi_paged_kv_append_int8(dims, to_dev_u16(q, device), to_dev_u16(k, device), to_dev_u16(v, device),
                                      torch.from_numpy(table).to(device), table.shape[0], bt_d, cl_d,
                                      to_dev_i32(slots, device), qo, k8, v8, ka, va, ko, vo, err) == 0
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(dims) // 4 + 4, dtype=torch.float32, device=device)
    assert mi.mi_paged_decode_attention_int8(dims, qo, k8, v8, ka, va, bt_d, cl_d, 0.09, out, ws, dev_err=err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    host = {"k8": k8.cpu().numpy(), "v8": v8.cpu().numpy(),
            "k_amax": ka.cpu().numpy().reshape(nb, Hkv), "v_amax": va.cpu().numpy().reshape(nb, Hkv),
            "k_open": from_dev_u16(ko), "v_open": from_dev_u16(vo)}
    return from_dev_u16(qo), from_dev_u16(out), host


def test_int8_swap_round_trip_keeps_the_next_step_bitwise(cuda_device):
    import torch
    mi = _mi()
    lens = [300, 127, 64, 1000, 45]
    Hq, Hkv, d = 8, 2, 128
    r, st, bt, slots, q, k, v, free = _int8_batch(11, lens, Hq, Hkv, d)
    nb = st["k8"].shape[0]
    cl = np.array(lens, np.int32) + 1
    table = oracle.rope_table(1e6, d, 2048)
    q_ref, out_ref, after_ref = _step(mi, cuda_device, st, bt, cl, slots, q, k, v, Hq, table)

    # swap sequence 3 out: its blocks (codes and maxima) and its open slot
    s = 3
    nbs = -(-int(cl[s]) // BS)
    old = bt[s, :nbs].copy()
    dev = {key: torch.from_numpy(st[key].copy()).to(cuda_device) for key in ("k8", "v8", "k_amax", "v_amax")}
    dev["k_open"], dev["v_open"] = to_dev_u16(st["k_open"], cuda_device), to_dev_u16(st["v_open"], cuda_device)
    row = {"k8": Hkv * BS * d, "v8": Hkv * BS * d, "k_amax": Hkv * 4, "v_amax": Hkv * 4,
           "k_open": Hkv * 64 * d * 2, "v_open": Hkv * 64 * d * 2}
    count = {"k8": nb, "v8": nb, "k_amax": nb, "v_amax": nb, "k_open": st["k_open"].shape[0],
             "v_open": st["v_open"].shape[0]}
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    host = {}
    for key in dev:
        n_out = 1 if key.endswith("open") else nbs
        src_ids = np.array([slots[s]], np.int32) if key.endswith("open") else old
        host[key] = torch.empty((n_out, row[key]), dtype=torch.uint8).pin_memory()
        assert mi.mi_kv_copy_rows(dev[key], count[key], to_dev_i32(src_ids, cuda_device), host[key], n_out,
                                  to_dev_i32(np.arange(n_out, dtype=np.int32), cuda_device), n_out, row[key],
                                  err) == 0
    torch.cuda.synchronize()
    # the freed blocks and slot are reused meanwhile: overwrite them
    for key in ("k8", "v8"):
        dev[key][torch.from_numpy(old.astype(np.int64)).to(cuda_device)] = 77
    for key in ("k_amax", "v_amax"):
        dev[key][torch.from_numpy(old.astype(np.int64)).to(cuda_device)] = float("nan")
    for key in ("k_open", "v_open"):
        dev[key][int(slots[s])] = float("nan")
    # swap in: fresh blocks and another slot
    new = np.asarray(free[:nbs], np.int32)
    new_slot = np.int32(len(lens))                    # a slot nobody used
    for key in dev:
        n_in = 1 if key.endswith("open") else nbs
        dst_ids = np.array([new_slot], np.int32) if key.endswith("open") else new
        assert mi.mi_kv_copy_rows(host[key], n_in, to_dev_i32(np.arange(n_in, dtype=np.int32), cuda_device),
                                  dev[key], count[key], to_dev_i32(dst_ids, cuda_device), n_in, row[key], err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    moved = {key: dev[key].cpu().numpy() for key in ("k8", "v8", "k_amax", "v_amax")}
    moved["k_open"], moved["v_open"] = from_dev_u16(dev["k_open"]), from_dev_u16(dev["v_open"])
    bt2, slots2 = bt.copy(), slots.copy()
    bt2[s, :nbs] = new
    slots2[s] = new_slot
    q2, out2, after2 = _step(mi, cuda_device, moved, bt2, cl, slots2, q, k, v, Hq, table)
    assert np.array_equal(q2, q_ref) and np.array_equal(out2, out_ref)
    # the moved sequence's state after the step, at its new place, equals the unmoved one's
    for key in ("k8", "v8", "k_amax", "v_amax"):
        assert np.array_equal(after2[key][new], after_ref[key][old]), key
    for key in ("k_open", "v_open"):
        assert np.array_equal(after2[key][new_slot], after_ref[key][slots[s]]), key
