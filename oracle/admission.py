"""Admission rule of the SLO-aware, KV-cache-protecting scheduler (test
infrastructure only).

Restates the three-level brake of the GitLink project report
"mxdyymxgxtlkjdxtjyhysx" (section "我们的解决方案：SLO感知与KV Cache保护调度器",
"基于实时状态的‘三等级刹车’决策机制"), read as a decision on whether a new
prefill request may enter, taken from the KV-cache pool's free space:

  1. hard brake: the free share of the pool is below the hard threshold
     (the report's example: 10%) -> no new prefill, whatever is running;
  2. soft brake: at least one decode is running and the free share is below
     the safe threshold (example: 30%) -> no new prefill for now;
  3. proceed: otherwise.

"Below" is read as strictly less than. Thresholds are given in basis points
(1/10000) of the pool and compared exactly in integers:
free / total < bp / 10000  <=>  free * 10000 < bp * total.
"""
from __future__ import annotations

PROCEED, SOFT_BRAKE, HARD_BRAKE = 0, 1, 2
HARD_BP, SOFT_BP = 1000, 3000  # the report's example thresholds: 10% and 30%


def below(free: int, total: int, bp: int) -> bool:
    """free / total < bp / 10000, exactly."""
    return free * 10000 < bp * total


def admission(num_free: int, num_blocks: int, running_decodes: int, hard_bp: int = HARD_BP,
              soft_bp: int = SOFT_BP) -> int:
    """The brake level for one new prefill request."""
    assert num_blocks >= 1 and 0 <= num_free <= num_blocks and running_decodes >= 0
    if below(num_free, num_blocks, hard_bp):
        return HARD_BRAKE
    if running_decodes > 0 and below(num_free, num_blocks, soft_bp):
        return SOFT_BRAKE
    return PROCEED
