"""The backward's static per-CTA schedule of its work list (host only).

Plans and one-shot calls of the backward lay its longest-first work list out
per CTA by list scheduling: each item goes, in list order, to the CTA that
is free first.  These tests check what the schedule promises, on the five
workloads, the candidate workload and random lists: it is a partition of the
items; no CTA ends more than one item past the mean (the list-scheduling
bound); replayed in list order the assignment is the free-first one; and a
CTA's items keep the list's order.
"""
import numpy as np
import pytest

from hstu_jagged_attention_gb300 import binding, workloads
from oracle import worklist

GRID = 152
MIB = 1 << 20


def bwd_cost(items, hist=None):
    nq = (items[:, 1] + 127) // 128
    h = items[:, 1] if hist is None else hist
    return np.where(128 * items[:, 3] >= h, 1, nq - items[:, 3])


def lists():
    out = []
    for name in workloads.WORKLOAD_NAMES:
        w = workloads.workload(name)
        ib = worklist.items_bwd(w.offsets, w.heads)
        out.append((name, ib, bwd_cost(ib)))
    w, nt = workloads.candidate_workload()
    ib, hb = worklist.items_bwd_targets(w.offsets, nt, w.heads)
    out.append(("candidates", ib, bwd_cost(ib, hb)))
    return out


LISTS = lists()


def replay_free_first(cost, grid):
    """Owner of each item when each goes, in list order, to the CTA with the
    least load so far (ties: the lower CTA)."""
    load = np.zeros(grid, dtype=np.int64)
    owner = np.empty(len(cost), dtype=np.int64)
    for i in range(len(cost)):
        c = int(np.argmin(load))  # argmin takes the lowest index among ties
        owner[i] = c
        load[c] += cost[i] + 1
    return owner, int(load.max())


def check(cost, grid):
    order, first, span = binding.hstu_worklist_schedule(cost, grid)
    assert sorted(order.tolist()) == list(range(len(cost)))
    assert first[0] == 0 and first[-1] == len(cost) and np.all(np.diff(first) >= 0)
    owner = np.empty(len(cost), dtype=np.int64)
    for c in range(grid):
        seg = order[first[c]:first[c + 1]]
        assert np.all(np.diff(seg) > 0)  # the list's order within a CTA
        owner[seg] = c
    want, want_span = replay_free_first(cost, grid)
    assert np.array_equal(owner, want)
    assert span == want_span
    # list scheduling: the last item of the longest CTA started when that CTA
    # was the least loaded, so at or before the mean
    assert span <= (cost + 1).sum() / grid + (cost + 1).max()
    return span


@pytest.mark.parametrize("name,items,cost", LISTS, ids=[x[0] for x in LISTS])
def test_schedule_is_free_first_list_scheduling(name, items, cost):
    grid = min(GRID, len(items))
    span = check(cost, grid)
    # close to the mean on these workloads (longest first)
    assert span <= 1.02 * (cost + 1).sum() / grid + 2, name


@pytest.mark.parametrize("seed", range(8))
def test_schedule_random_lists(seed):
    rng = np.random.default_rng(300 + seed)
    lengths = rng.integers(0, 9000, size=int(rng.integers(1, 120)))
    heads = int(rng.integers(1, 5))
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    items = worklist.items_bwd(off, heads)
    if len(items) == 0:
        return
    cost = bwd_cost(items)
    grid = int(rng.integers(1, min(200, len(items)) + 1))
    span = check(cost, grid)
    order, first, _ = binding.hstu_worklist_schedule(cost, grid)
    order2, first2, span2 = binding.hstu_worklist_schedule(cost, grid)
    assert np.array_equal(order, order2) and np.array_equal(first, first2) and span == span2


def test_schedule_hand_case():
    # costs 5, 3, 3, 2, 1, 1 on 2 CTAs (units = cost + 1): CTA 0 takes item 0
    # (6), CTA 1 items 1 (4) and 2 (8); CTA 0 then item 3 (9); CTA 1 item 4
    # (10); CTA 0 item 5 (11)
    order, first, span = binding.hstu_worklist_schedule(np.array([5, 3, 3, 2, 1, 1]), 2)
    assert first.tolist() == [0, 3, 6]
    assert order.tolist() == [0, 3, 5, 1, 2, 4]
    assert span == 11


def test_schedule_rejects_bad_arguments():
    cost = np.array([3, 2, 1], dtype=np.int32)
    for grid in (0, 4):
        with pytest.raises(binding.HstuError):
            binding.hstu_worklist_schedule(cost, grid)
    with pytest.raises(binding.HstuError):
        binding.hstu_worklist_schedule(np.array([3, 0, 1]), 2)
