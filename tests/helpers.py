"""Shared test plumbing: run a workload's decode step through the library's
C ABI (device side) and through the oracle (host side) on the same inputs.

Nothing here computes a result of the method: the library and the oracle do.
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle.pool import PoolModel
from workloads import (WORKLOADS, context_lengths, history_cache, initial_free_order,
                       new_token_values, setup_pool)

MAX_ABS_TOL = 1e-2   # attention: max |gpu - fp64 oracle| for bf16 inputs, unit-variance V
MEAN_ABS_TOL = 1e-3  # attention: mean |gpu - fp64 oracle|


def pools_for(w):
    """(library pool, oracle pool model) after the workload's history, plus ctx."""
    import paged_kv_decode_25_gb300 as mi
    ctx = context_lengths(w)
    order = initial_free_order(w)
    lib = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    model = PoolModel(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    setup_pool(w, lib, ctx)
    setup_pool(w, model, ctx)
    return lib, model, ctx


def grow(pool, B, new_len):
    for b in range(B):
        assert pool.alloc(b, int(new_len[b])) == 0


def to_dev_u16(a, device):
    """uint16 numpy bits -> torch bfloat16 tensor on device (same bits)."""
    import torch
    return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)


def from_dev_u16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev_i32(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


def attn_errors(gpu_bits, ref):
    got = oracle.bf16_to_f64(gpu_bits)
    err = np.abs(got - ref)
    return float(err.max()), float(err.mean())


def assert_attention_close(gpu_bits, ref, what=""):
    mx, mean = attn_errors(gpu_bits, ref)
    assert np.all(np.isfinite(oracle.bf16_to_f64(gpu_bits))), what
    assert mx <= MAX_ABS_TOL and mean <= MEAN_ABS_TOL, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def gather_used_blocks(kc_d, vc_d, bt, cl, rows=None):
    """Host copies of the cache blocks that requests `rows` (default: all) use
    within their first ceil(cl/16) table entries, renumbered 0..n-1, and their
    tables rewritten to the new numbers (-1 elsewhere). Only moves data: the
    oracle, not this helper, computes results over it."""
    import torch
    rows = list(range(len(cl))) if rows is None else list(rows)
    live = [bt[b, :-(-max(int(cl[b]), 0) // 16)] for b in rows]
    used = sorted({int(x) for row in live for x in row})
    remap = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.int64, device=kc_d.device)
    kc, vc = from_dev_u16(kc_d[idx]), from_dev_u16(vc_d[idx])
    bt_s = np.full((len(rows), bt.shape[1]), -1, np.int32)
    for i, row in enumerate(live):
        bt_s[i, :len(row)] = [remap[int(x)] for x in row]
    return kc, vc, bt_s, used
