"""The allocation-free attention entry point, through the C ABI.

mi_paged_decode_attention_noalloc serves callers that cannot call cudaMalloc
(a plugin whose host framework owns all device memory, a serving loop that
forbids allocator calls because they can synchronise the device, a process
held to a fixed device-memory budget): its split-KV partials live in a fixed
array inside the library. This file is collected last so that a run stopping
at its first failure has already run every other test; it also passes when
run alone in a fresh process.
"""
import numpy as np
import pytest

from helpers import MAX_ABS_TOL, MEAN_ABS_TOL, from_dev_u16, to_dev_i32, to_dev_u16
from workloads import BLOCK, CANARY_BF16, bf16_normal

pytestmark = pytest.mark.gpu


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _paged_case(seed, B=24, Hq=32, Hkv=8, d=128):
    """Random paged caches whose units span several CTAs (so the scratch holds
    real partials), plus two different query batches."""
    r = np.random.Generator(np.random.PCG64(seed))
    lens = np.floor(np.exp(r.uniform(np.log(17), np.log(6000), size=B))).astype(np.int32)
    lens[:3] = [1, 0, 16]
    nblk = [-(-max(int(n), 0) // BLOCK) for n in lens]
    nb = sum(nblk) + 11
    mbps = max(nblk)
    perm = r.permutation(nb)
    bt = np.full((B, mbps), -1, np.int32)
    kc = np.full((nb, Hkv, BLOCK, d), CANARY_BF16, np.uint16)
    vc = kc.copy()
    i = 0
    for b, n in enumerate(lens):
        for j in range(nblk[b]):
            blk = int(perm[i]); i += 1
            bt[b, j] = blk
            m = min(BLOCK, int(n) - j * BLOCK)
            kc[blk, :, :m] = bf16_normal(r, (Hkv, m, d))
            vc[blk, :, :m] = bf16_normal(r, (Hkv, m, d))
    q1 = bf16_normal(r, (B, Hq, d))
    q2 = bf16_normal(r, (B, Hq, d))
    return q1, q2, kc, vc, bt, lens, nb, mbps


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_device):
    import torch
    import paged_kv_decode_25_gb300 as mi
    q1, q2, kc, vc, bt, lens, nb, mbps = _paged_case(41)
    B, Hq, d = q1.shape
    Hkv = kc.shape[1]
    dims = mi.dims(B, Hq, Hkv, d, nb, mbps)
    assert 0 < mi.mi_paged_decode_workspace_bytes(dims) <= mi.MI_NOALLOC_SCRATCH_BYTES
    kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(lens, cuda_device)
    scale = 1.0 / np.sqrt(d)
    qs = [to_dev_u16(q, cuda_device) for q in (q1, q2)]

    # the existing entry point with a caller-allocated workspace
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(dims) // 4 + 4, dtype=torch.float32, device=cuda_device)
    refs = []
    for q_d in qs:
        out = torch.empty_like(q_d)
        assert mi.mi_paged_decode_attention(dims, q_d, kc_d, vc_d, bt_d, cl_d, scale, out, ws) == mi.MI_OK
        refs.append(out)
    torch.cuda.synchronize()

    # two allocation-free calls in a row on the same stream
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    outs = [torch.full_like(q_d, float("nan")) for q_d in qs]
    for q_d, out in zip(qs, outs):
        st = mi.mi_paged_decode_attention_noalloc(dims, q_d, kc_d, vc_d, bt_d, cl_d, scale, out, dev_err=err)
        assert st == mi.MI_OK, mi.status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for ref, out in zip(refs, outs):
        # the same kernel on the same grid and split: the same bits
        assert np.array_equal(from_dev_u16(out), from_dev_u16(ref))
        a, b = _f32(from_dev_u16(out)), _f32(from_dev_u16(ref))
        assert np.all(np.isfinite(a))
        diff = np.abs(a - b)
        assert diff.max() <= MAX_ABS_TOL and diff.mean() <= MEAN_ABS_TOL, (diff.max(), diff.mean())
    # the two calls saw different queries, so their outputs differ
    assert not np.array_equal(from_dev_u16(outs[0]), from_dev_u16(outs[1]))


def test_noalloc_rejects_what_it_cannot_serve(cuda_device):
    import paged_kv_decode_25_gb300 as mi
    z = 16  # never dereferenced: every case is refused before anything is queued
    assert mi.mi_paged_decode_attention_noalloc(mi.dims(2, 18, 2, 128, 8, 4), z, z, z, z, z, 1.0, z) \
        == mi.MI_ERR_UNSUPPORTED   # G = 9
    assert mi.mi_paged_decode_attention_noalloc(mi.dims(2, 8, 2, 96, 8, 4), z, z, z, z, z, 1.0, z) \
        == mi.MI_ERR_UNSUPPORTED   # head_dim 96
    assert mi.mi_paged_decode_attention_noalloc(mi.dims(0, 8, 2, 128, 8, 4), None, None, None, None, None, 1.0,
                                                None) == mi.MI_OK
