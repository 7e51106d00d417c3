"""The split plan that each CTA of the decode attention keeps in the workspace
for the next launch is used only when it is this CTA's and intact.

* A workspace handed over at a shifted address (512 bytes: two entries at
  this batch size) over memory that still holds the entries of a launch with
  the same dims and lengths: every CTA then finds another CTA's entry at its
  position. The output must be bit for bit the fresh launch's, and match the
  oracle.
* An entry whose cached plan words were changed after it was written (its key
  and lengths intact): the same.
Both cases happen when a caller frees a workspace and allocates another,
which a caching allocator may place over the old one at another offset, or
uses one buffer as the workspace of different dims."""
import numpy as np
import pytest

import oracle
from helpers import assert_attention_close, from_dev_u16, to_dev_i32, to_dev_u16
from workloads import BLOCK, bf16_normal

pytestmark = pytest.mark.gpu

PLAN_MAGIC = 0x6E616C50


def _case(seed, d_head=64, Hq=7, Hkv=7):
    r = np.random.Generator(np.random.PCG64(seed))
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 200, 1000, 4097]
    B = len(lens)
    nblk = [-(-n // BLOCK) for n in lens]
    nb = sum(nblk) + 3
    perm = r.permutation(nb)
    bt = np.full((B, max(nblk) + 1), -1, np.int32)
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    kc = bf16_normal(r, (nb, Hkv, BLOCK, d_head))
    vc = bf16_normal(r, (nb, Hkv, BLOCK, d_head))
    q = bf16_normal(r, (B, Hq, d_head))
    return q, kc, vc, bt, np.array(lens, np.int32)


def _attend(mi, d, q_d, kc_d, vc_d, bt_d, cl_d, ws_view, device):
    import torch
    out = torch.full(q_d.shape, float("nan"), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    st = mi.mi_paged_decode_attention(d, q_d, kc_d, vc_d, bt_d, cl_d, 0.09, out, ws_view,
                                      workspace_bytes=ws_view.numel() * 4, dev_err=err)
    assert st == 0, mi.status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return from_dev_u16(out)


def _setup(device):
    import torch
    import paged_kv_decode_25_gb300 as mi
    q, kc, vc, bt, cl = _case(7)
    B, Hq, d_head = q.shape
    d = mi.dims(B, Hq, kc.shape[1], d_head, kc.shape[0], bt.shape[1])
    n = mi.mi_paged_decode_workspace_bytes(d)
    assert n > 0
    big = torch.zeros(n // 4 + 1024, dtype=torch.float32, device=device)  # room for a 4 KB shift
    ref = oracle.paged_attention(q, kc, vc, bt, cl, 0.09, nthreads=8)
    args = (to_dev_u16(q, device), to_dev_u16(kc, device), to_dev_u16(vc, device), to_dev_i32(bt, device),
            to_dev_i32(cl, device))
    return mi, d, n, big, ref, args


def test_plan_entries_of_other_ctas_are_not_used(cuda_device):
    mi, d, n, big, ref, args = _setup(cuda_device)
    first = _attend(mi, d, *args, big[: n // 4], cuda_device)
    assert_attention_close(first, ref, "fresh workspace")
    again = _attend(mi, d, *args, big[: n // 4], cuda_device)          # its own entries: reused
    assert np.array_equal(first, again)
    for shift_floats in (128, 64, 1024):                                # 512 B, 256 B, 4 KB
        shifted = _attend(mi, d, *args, big[shift_floats: shift_floats + n // 4], cuda_device)
        assert np.array_equal(first, shifted), shift_floats


def test_damaged_plan_entries_are_not_used(cuda_device):
    import torch
    mi, d, n, big, ref, args = _setup(cuda_device)
    ws = big[: n // 4]
    first = _attend(mi, d, *args, ws, cuda_device)
    words = ws.view(torch.int32)
    starts = torch.nonzero(words == PLAN_MAGIC).flatten()
    starts = starts[starts + 14 < words.numel()]
    assert starts.numel() > 0                                           # the entries were written
    # bump the low word of each entry's cached TC (words 12-13 of the entry:
    # key[8], P, sum, TB, TC, range plan)
    words[starts + 12] += 1
    torch.cuda.synchronize()
    second = _attend(mi, d, *args, ws, cuda_device)
    assert np.array_equal(first, second)
    assert_attention_close(second, ref, "damaged entries")
