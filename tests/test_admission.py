"""mi_kv_pool_admission against the oracle's brake rule (exact, host only),
and a continuous-batching schedule driven through the library pool and
through the oracle's pool model: identical event traces, and the brakes keep
running decodes from being preempted on a load that preempts without them."""
import os

import numpy as np
import pytest

from oracle import admission as A
from oracle.pool import PoolModel
from workloads import serving_churn


@pytest.fixture(scope="module")
def mi():
    import paged_kv_decode_25_gb300 as m
    from paged_kv_decode_25_gb300 import build
    build.build()
    return m


def _pool_with_free(mi, total, free):
    p = mi.Pool(total, 2, total)
    if free < total:
        assert p.alloc(0, (total - free) * 16) == 0
    assert p.num_free() == free
    return p


def test_golden_table_through_the_library(mi):
    path = os.path.join(os.path.dirname(__file__), "golden", "admission_brakes.txt")
    names = {"proceed": mi.MI_ADMIT_PROCEED, "soft": mi.MI_ADMIT_SOFT_BRAKE, "hard": mi.MI_ADMIT_HARD_BRAKE}
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            free, total, running, want = int(line[0]), int(line[1]), int(line[2]), names[line[3]]
            p = _pool_with_free(mi, total, free)
            assert p.admission(running) == want, line
            p.close()
            n += 1
    assert n >= 15


def test_library_matches_oracle_on_random_states(mi):
    r = np.random.Generator(np.random.PCG64(3))
    for _ in range(300):
        total = int(r.integers(1, 300))
        free = int(r.integers(0, total + 1))
        p = _pool_with_free(mi, total, free)
        for _ in range(5):
            running = int(r.integers(0, 3))
            hard, soft = (int(x) for x in r.integers(0, 10001, size=2))
            assert p.admission(running, hard, soft) == A.admission(free, total, running, hard, soft)
        p.close()


def test_admission_errors(mi):
    p = mi.Pool(8, 2, 8)
    assert mi.mi_kv_pool_admission(p.handle, -1)[0] == mi.MI_ERR_INVALID_ARG
    assert mi.mi_kv_pool_admission(p.handle, 0, 10001, 0)[0] == mi.MI_ERR_INVALID_ARG
    assert mi.mi_kv_pool_admission(p.handle, 0, 0, -1)[0] == mi.MI_ERR_INVALID_ARG
    assert mi.mi_kv_pool_admission(None, 0)[0] == mi.MI_ERR_INVALID_ARG


@pytest.mark.parametrize("brakes", [True, False])
def test_churn_trace_matches_oracle(mi, brakes):
    lib, model = mi.Pool(2048, 4096, 256), PoolModel(2048, 4096, 256)
    a = serving_churn(lib, 400, 1, use_brakes=brakes)
    b = serving_churn(model, 400, 1, use_brakes=brakes)
    assert a == b


def test_brakes_prevent_preemption_on_a_heavy_load(mi):
    runs = {}
    for brakes in (True, False):
        lib = mi.Pool(2048, 4096, 256)
        t = serving_churn(lib, 400, 1, use_brakes=brakes)
        runs[brakes] = (sum(len(x[1]) for x in t), sum(len(x[2]) for x in t))
    assert runs[False][0] > 0          # without brakes running decodes get preempted
    assert runs[True][0] == 0          # with them none is
    assert runs[True][1] >= runs[False][1]
