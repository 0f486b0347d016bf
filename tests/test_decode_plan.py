"""The decode attention's split plan (host logic, no GPU): how a decode step's
(sequence, rank, kv head) units are cut into work items for the persistent
kernel.  A decode step is bounded below by the time to read memory ("Tensor
parallelism from scratch", "The cost of communication"), and the decode
attention reads the KV cache, so the plan's job is to keep every pipeline
streaming until the cache has been read: these tests pin its
structure and check, on a list-scheduling model of the pipelines, that the cut
finishes no later than whole units would and close to the even share."""

import heapq
import itertools
import math

import pytest

from tensor_transformer_forward_gb300 import binding
from tensor_transformer_forward_gb300.binding import TPError

BK = 128          # keys per tile of the tensor-core decode kernel
WANT = (1, 2, 4, 8)  # split counts the levels aim at


def plan(kv, units, sms, hd=128, group=2, max_splits=64):
    return binding.tp_debug_decode_plan(kv, units, sms, hd, group, max_splits)


GRID = list(itertools.product((1, 17, 128, 129, 2049, 4097, 32769),   # max_kv_len
                              (1, 7, 64, 512, 1024, 5000),            # units
                              (148, 152),                             # SMs
                              (64, 128),                              # head_dim
                              (1, 2, 8),                              # q heads per kv head
                              (1, 3, 8, 64)))                         # splits the workspace holds


@pytest.mark.parametrize("kv,units,sms,hd,group,max_splits", GRID)
def test_plan_structure(kv, units, sms, hd, group, max_splits):
    u, s = plan(kv, units, sms, hd, group, max_splits)
    assert len(u) == len(s) == 4
    assert sum(u) == units and min(u) >= 0
    assert all(1 <= x <= max(1, min(max_splits, 64)) for x in s)
    nt = math.ceil(kv / BK)
    if hd != 128 or s[0] != 1:
        # one level: every unit split alike
        assert u[0] == units and u[1:] == [0, 0, 0]
        if hd == 128:
            assert s[0] <= nt  # no split without a key tile
        return
    used = [l for l in range(4) if u[l] > 0]
    # levels are taken in order and cut finer as the work runs out
    assert [s[l] for l in used] == sorted(s[l] for l in used)
    for l in used:
        assert s[l] <= min(WANT[l], max_splits, nt)
        chunk = math.ceil(nt / s[l])
        assert (s[l] - 1) * chunk < nt  # every split of a full-length unit holds key tiles


def test_plan_rejects_bad_arguments():
    for args in [(0, 8, 152, 128, 2, 64), (2049, 0, 152, 128, 2, 64), (2049, 8, 0, 128, 2, 64),
                 (2049, 8, 152, 96, 2, 64), (2049, 8, 152, 128, 3, 64), (2049, 8, 152, 128, 2, 0)]:
        with pytest.raises(TPError):
            binding.tp_debug_decode_plan(*args)


def _items(kv, u, s):
    """Key tiles of every item in hand-out order (a split of a full-length unit)."""
    nt = math.ceil(kv / BK)
    out = []
    for l in range(4):
        chunk = math.ceil(nt / s[l])
        for _ in range(u[l]):
            out.extend(max(0, min(chunk, nt - k * chunk)) for k in range(s[l]))
    return out


def _makespan(costs, pipes):
    heap = [0.0] * pipes
    for c in costs:
        heapq.heappush(heap, heapq.heappop(heap) + c)
    return max(heap)


# (max_kv_len, units, SMs, q heads per kv head): the decode configurations'
# attention (128 x 2049 keys and 64 x 4097 at tp 2, 32 x 2049 at tp 16) and the
# mixed step's decode beside a prefill (95 SMs), plus short and long contexts
CASES = [(2049, 1024, 152, 2), (4097, 512, 152, 2), (2049, 512, 152, 8), (2049, 1024, 95, 2),
         (129, 5000, 152, 2), (32769, 64, 152, 2), (1025, 2000, 148, 4)]


@pytest.mark.parametrize("kv,units,sms,group", CASES)
def test_plan_finishes_no_later_than_whole_units(kv, units, sms, group):
    """Pipelines (two per SM) take the next item when they run dry; an item costs
    its key tiles plus one tile's worth of start-up.  The plan's items never
    finish later than whole units would, and stay within a unit's worth of
    the even share of the work."""
    u, s = plan(kv, units, sms, 128, group)
    items = _items(kv, u, s)
    nt = math.ceil(kv / BK)
    assert sum(items) == units * nt  # the splits cover every key tile once
    pipes = 2 * sms
    cut = _makespan([t + 1.0 for t in items], pipes)
    whole = _makespan([nt + 1.0] * units, pipes)
    even = sum(t + 1.0 for t in items) / pipes
    assert cut <= whole + 1e-9
    assert cut <= even + nt + 1.0


def test_plan_mixed_step_decode_within_five_percent_of_even_share():
    # 128 decode sequences x 2 ranks x 4 kv heads, 2049 keys, all 152 SMs
    u, s = plan(2049, 1024, 152, 128, 2)
    items = _items(2049, u, s)
    cut = _makespan([t + 1.0 for t in items], 304)
    even = sum(t + 1.0 for t in items) / 304
    assert cut <= 1.05 * even
    assert u[1:] != [0, 0, 0]  # whole units alone would leave the last pipelines idle
