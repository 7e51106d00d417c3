"""The multi-GPU path is replicas only (requests are independent; no exchange
step on the hot path). Its host logic runs here as two CPU ranks over gloo:
the barrier, the max-over-ranks step time every rank agrees on, the
whole-job rate from it, and the reference arm doing no work on rank 1."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from workloads import WORKLOADS
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_setup(None)
        assert (r, w, local) == (rank, world, rank)
        bench.barrier(world)
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower replica
        ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        rate = bench.whole_job_rate(1000.0, ms * 1e-3, world)

        class A:
            steps, warmup, gpus = 1, 0, world
        # the reference arm: rank 0 alone runs and prints; the others return at once
        out = None
        if rank != 0:
            out = bench.run_reference(A, WORKLOADS["tiny"], rank, world)
        bench.barrier(world)
        results[rank] = (ms, rate, out)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank, args=(2, _free_port(), results), nprocs=2, join=True, start_method="spawn")
        res = dict(results)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        ms, rate, out = res[rank]
        assert ms == 15.0                          # both ranks see the slowest rank's time
        assert rate == pytest.approx(2 * 1000.0 / 0.015)
    assert res[1][2] is None
