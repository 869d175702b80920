"""The static per-CTA schedule of a work list (host only, no GPU).

Plans and one-shot calls lay a longest-first work list out per CTA: each
item goes, in list order, to the CTA that is free first (list scheduling),
and where the streamed operands of all (sequence, head) groups exceed 48 MiB
the groups are taken in batches, so that the CTAs work on a few groups at a
time.  These tests check what the schedule promises, on the five workloads,
the candidate workload and random lists: it is a partition of the items; no
CTA ends more than one item past the mean (the list-scheduling bound); a
CTA's items keep the list's order within a batch; replayed in list order the
assignment is the free-first one; and the groups running at once stay few.
"""
import numpy as np
import pytest

from hstu_jagged_attention_gb300 import binding, workloads
from oracle import worklist

GRID = 152
MIB = 1 << 20


def fwd_cost(items, hist=None):
    if hist is None:
        return items[:, 3] + 1
    return np.minimum(items[:, 3], (hist + 127) // 128) + 1


def bwd_cost(items, hist=None):
    nq = (items[:, 1] + 127) // 128
    h = items[:, 1] if hist is None else hist
    return np.where(128 * items[:, 3] >= h, 1, nq - items[:, 3])


def lists():
    out = []
    for name in workloads.WORKLOAD_NAMES:
        w = workloads.workload(name)
        it = worklist.items(w.offsets, w.heads)
        out.append((f"{name}/fwd", it, fwd_cost(it), w.d))
        ib = worklist.items_bwd(w.offsets, w.heads)
        out.append((f"{name}/bwd", ib, bwd_cost(ib), w.d))
    w, nt = workloads.candidate_workload()
    it, hs = worklist.items_targets(w.offsets, nt, w.heads)
    out.append(("candidates/fwd", it, fwd_cost(it, hs), w.d))
    ib, hb = worklist.items_bwd_targets(w.offsets, nt, w.heads)
    out.append(("candidates/bwd", ib, bwd_cost(ib, hb), w.d))
    return out


LISTS = lists()


def timeline(items, cost, order, first):
    """(start, end, group, group bytes) of every item, CTA by CTA."""
    ev = []
    for c in range(len(first) - 1):
        t = 0
        for i in order[first[c]:first[c + 1]]:
            ev.append((t, t + int(cost[i]) + 1, (int(items[i, 0]), int(items[i, 2]))))
            t += int(cost[i]) + 1
    return ev


@pytest.mark.parametrize("name,items,cost,d", LISTS, ids=[x[0] for x in LISTS])
def test_schedule_partitions_and_bounds(name, items, cost, d):
    grid = min(GRID, len(items))
    order, first, span = binding.hstu_worklist_schedule(items, cost, d, grid)
    assert sorted(order.tolist()) == list(range(len(items)))
    assert first[0] == 0 and first[-1] == len(items) and np.all(np.diff(first) >= 0)
    loads = np.array([int((cost[order[first[c]:first[c + 1]]] + 1).sum()) for c in range(grid)])
    assert loads.max() == span
    # list scheduling: the last item of the longest CTA started when that CTA
    # was the least loaded, so it started at or before the mean
    assert span <= (cost + 1).sum() / grid + (cost + 1).max()
    # and in practice close to the mean on these workloads
    assert span <= 1.02 * (cost + 1).sum() / grid + 2, name


@pytest.mark.parametrize("name,items,cost,d", LISTS, ids=[x[0] for x in LISTS])
def test_schedule_groups_running_at_once_stay_few(name, items, cost, d):
    grid = min(GRID, len(items))
    order, first, _ = binding.hstu_worklist_schedule(items, cost, d, grid)
    ev = timeline(items, cost, order, first)
    seq_len = {(int(x[0]), int(x[2])): int(x[1]) for x in items}
    all_bytes = sum(n * d * 4 for n in seq_len.values())
    starts = sorted({s for s, _, _ in ev})
    worst = 0
    for t in starts[:: max(1, len(starts) // 100)]:
        running = {g for s, e, g in ev if s <= t < e}
        worst = max(worst, sum(seq_len[g] * d * 4 for g in running))
    if all_bytes > 48 * MIB:
        # batches of at most 48 MiB of operands; a CTA still finishing a
        # long item of the previous batch overlaps the next
        assert worst <= 2 * 48 * MIB + max(seq_len.values()) * d * 4, (name, worst / MIB)


def test_schedule_one_batch_is_free_first_in_list_order():
    # a list whose operands fit one batch: replaying the items in list order,
    # each goes to the CTA with the least load so far (ties: the lower CTA)
    rng = np.random.default_rng(7)
    lengths = rng.integers(1, 2000, size=40)
    assert lengths.sum() * 3 * 64 * 4 <= 48 * MIB  # one batch
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    items = worklist.items(off, 3)
    cost = fwd_cost(items)
    grid = 16
    order, first, span = binding.hstu_worklist_schedule(items, cost, 64, grid)
    owner = np.empty(len(items), dtype=np.int64)
    for c in range(grid):
        seg = order[first[c]:first[c + 1]]
        assert np.all(np.diff(seg) > 0)  # the list's order within a CTA
        owner[seg] = c
    load = np.zeros(grid, dtype=np.int64)
    for i in range(len(items)):
        c = int(np.argmin(load))  # argmin takes the lowest index among ties
        assert owner[i] == c, i
        load[c] += cost[i] + 1
    assert load.max() == span


def test_schedule_batches_keep_list_order_within_each_group():
    # the candidate forward is batched; a CTA's items of one group run in
    # the list's order (longest first)
    name, items, cost, d = next(x for x in LISTS if x[0] == "candidates/fwd")
    order, first, _ = binding.hstu_worklist_schedule(items, cost, d, GRID)
    for c in range(GRID):
        seg = order[first[c]:first[c + 1]]
        by_group = {}
        for i in seg:
            by_group.setdefault((int(items[i, 0]), int(items[i, 2])), []).append(int(i))
        for ids in by_group.values():
            assert ids == sorted(ids)


@pytest.mark.parametrize("seed", range(6))
def test_schedule_random_lists(seed):
    rng = np.random.default_rng(300 + seed)
    lengths = rng.integers(0, 9000, size=int(rng.integers(1, 120)))
    heads = int(rng.integers(1, 5))
    d = int(rng.choice([32, 64, 128]))
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    items = worklist.items(off, heads)
    if len(items) == 0:
        return
    cost = fwd_cost(items)
    grid = int(rng.integers(1, min(200, len(items)) + 1))
    order, first, span = binding.hstu_worklist_schedule(items, cost, d, grid)
    assert sorted(order.tolist()) == list(range(len(items)))
    assert span <= (cost + 1).sum() / grid + (cost + 1).max()
    # deterministic
    order2, first2, span2 = binding.hstu_worklist_schedule(items, cost, d, grid)
    assert np.array_equal(order, order2) and np.array_equal(first, first2) and span == span2


def test_schedule_rejects_bad_arguments():
    items = worklist.items(np.array([0, 300], dtype=np.int32), 1)
    cost = fwd_cost(items)
    for grid in (0, len(items) + 1):
        with pytest.raises(binding.HstuError):
            binding.hstu_worklist_schedule(items, cost, 64, grid)
    with pytest.raises(binding.HstuError):
        binding.hstu_worklist_schedule(items, np.zeros_like(cost), 64, 1)
    with pytest.raises(binding.HstuError):
        binding.hstu_worklist_schedule(items, cost, 0, 1)
