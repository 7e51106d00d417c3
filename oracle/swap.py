"""Block copies between paged KV caches (test infrastructure only).

A swap-out moves whole KV blocks of a sequence from the device cache to a
cache in host memory, a swap-in moves them back into freshly allocated blocks
(NJU course brief "端侧大模型推理框架", optional task 3 "KV Cache Offloading":
inactive KV blocks are moved to CPU memory and brought back when needed). A
block is every KV head's 16 token rows, so a copy is the plain assignment
dst[dst_ids[i]] = src[src_ids[i]] for each listed pair, for K and V alike.
"""
from __future__ import annotations

import numpy as np


def copy_blocks(src: np.ndarray, src_ids, dst: np.ndarray, dst_ids) -> None:
    """dst[dst_ids[i]] = src[src_ids[i]] for every i, in order (in place)."""
    assert len(src_ids) == len(dst_ids)
    for a, b in zip(src_ids, dst_ids):
        dst[int(b)] = src[int(a)]
