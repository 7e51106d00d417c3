"""Pins for the oracle's admission rule: the hand-worked table of
tests/golden/admission_brakes.txt (the report's 10% / 30% example
thresholds), and invariants any reading of the rule must keep: the hard brake
ignores running decodes, no running decode never soft-brakes, more free blocks
never tighten the decision and more running decodes never loosen it."""
import os

import numpy as np

from oracle import admission as A

NAMES = {"proceed": A.PROCEED, "soft": A.SOFT_BRAKE, "hard": A.HARD_BRAKE}


def _golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "admission_brakes.txt")
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                rows.append((int(line[0]), int(line[1]), int(line[2]), NAMES[line[3]]))
    return rows


def test_hand_worked_table():
    rows = _golden()
    assert len(rows) >= 15
    for free, total, running, want in rows:
        assert A.admission(free, total, running) == want, (free, total, running)


def test_invariants_on_random_states():
    r = np.random.Generator(np.random.PCG64(21))
    for _ in range(3000):
        total = int(r.integers(1, 5000))
        free = int(r.integers(0, total + 1))
        running = int(r.integers(0, 4))
        hard, soft = sorted(int(x) for x in r.integers(0, 10001, size=2))
        d = A.admission(free, total, running, hard, soft)
        if d == A.HARD_BRAKE:
            assert all(A.admission(free, total, k, hard, soft) == A.HARD_BRAKE for k in range(4))
        if running == 0:
            assert d != A.SOFT_BRAKE
        if free < total:
            assert A.admission(free + 1, total, running, hard, soft) <= d
        assert A.admission(free, total, running + 1, hard, soft) >= d


def test_zero_thresholds_never_brake_and_full_thresholds_always_do():
    for total in (1, 7, 100):
        for free in range(total + 1):
            assert A.admission(free, total, 3, 0, 0) == A.PROCEED
            assert A.admission(free, total, 0, 10000, 10000) == (A.HARD_BRAKE if free < total else A.PROCEED)
