"""Plain Python enumeration of the attention work items.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

A work item is one block of BLOCK_M = 128 query rows of one (sequence, head).
Query block qt of sequence b needs the key blocks kt = 0..qt: the blocks
with kt > qt are entirely above the causal diagonal and are skipped, the
block kt = qt is the triangular one (ai6s.net "HSTU fused operator" post,
section 3.2, the three block-mask cases), so an item costs qt + 1 key
blocks.  Items are ordered longest first: cost descending, then b, h, qt
ascending.  Empty sequences contribute no items (section 4.2, jagged storage).

Each item is four int32: (first token of the sequence, sequence length,
head, qt).

With candidates (HSTU paper section 3.4 and Appendix H, Algorithm 1: the
M-FALCON mask), the last num_targets[b] tokens of sequence b see the
history and themselves only.  With hist = n - num_targets[b] and
KH = ceil(hist / 128) the key blocks that hold history keys, query block qt
needs key blocks 0 .. min(qt, KH) - 1 and its diagonal block qt: a block
strictly between them holds only keys of other candidates, which no row of
the query block sees.  Such an item costs min(qt, KH) + 1 key blocks, and
items_targets also returns each item's hist.

The forward on CTA pairs takes two consecutive query blocks, 2 qp and
2 qp + 1, of a (sequence, head) together: the pair walks the key blocks
0 .. min(2 qp + 1, nq - 1) (nq = ceil(n / 128)), so a pair item costs
min(2 qp + 2, nq) key blocks; items_pairs lists (first token, length,
head, qp) by cost descending, then b, h, qp ascending.
"""
from __future__ import annotations

import numpy as np

BLOCK_M = 128


def items(offsets, heads: int, block_m: int = BLOCK_M) -> np.ndarray:
    offsets = [int(x) for x in offsets]
    rows = []
    for b in range(len(offsets) - 1):
        n = offsets[b + 1] - offsets[b]
        tiles = (n + block_m - 1) // block_m
        for h in range(heads):
            for qt in range(tiles):
                rows.append((-(qt + 1), b, h, qt, offsets[b], n))
    rows.sort()
    out = np.array([(s0, n, h, qt) for (_, b, h, qt, s0, n) in rows], dtype=np.int32)
    return out.reshape(-1, 4)


def items_targets(offsets, num_targets, heads: int, block_m: int = BLOCK_M):
    """(items (n, 4) int32, hist (n,) int32), ordered by cost descending,
    then b, h, qt ascending."""
    offsets = [int(x) for x in offsets]
    rows = []
    for b in range(len(offsets) - 1):
        n = offsets[b + 1] - offsets[b]
        hist = n - int(num_targets[b])
        kh = (hist + block_m - 1) // block_m
        tiles = (n + block_m - 1) // block_m
        for h in range(heads):
            for qt in range(tiles):
                cost = min(qt, kh) + 1
                rows.append((-cost, b, h, qt, offsets[b], n, hist))
    rows.sort()
    it = np.array([(s0, n, h, qt) for (_, b, h, qt, s0, n, _hist) in rows], dtype=np.int32)
    hs = np.array([hist for (*_, hist) in rows], dtype=np.int32)
    return it.reshape(-1, 4), hs



def items_candidates(offsets, num_targets, heads: int, block_m: int = BLOCK_M):
    """The candidates-only work list: the items of items_targets whose query
    block holds a candidate row (rows hist .. n-1 of a sequence with at least
    one candidate), in the same order."""
    it, hs = items_targets(offsets, num_targets, heads, block_m)
    keep = [r for r in range(len(hs))
            if hs[r] < it[r, 1] and any(hs[r] <= i < it[r, 1]
                                        for i in range(it[r, 3] * block_m, (it[r, 3] + 1) * block_m))]
    return it[keep].reshape(-1, 4), hs[keep]


def items_bwd_targets(offsets, num_targets, heads: int, block_m: int = BLOCK_M):
    """The backward's work list with candidates: (items (n, 4), hist (n,)).
    Key block kt is seen by the query blocks that hold a row seeing one of
    its keys: a history key by every later row, a candidate key by its own
    row only.  So the item walks query blocks kt .. last when the block has
    a history key, else block kt alone; cost descending, then b, h, kt."""
    offsets = [int(x) for x in offsets]
    rows = []
    for b in range(len(offsets) - 1):
        n = offsets[b + 1] - offsets[b]
        hist = n - int(num_targets[b])
        nq = (n + block_m - 1) // block_m
        for h in range(heads):
            for kt in range(nq):
                has_history_key = any(j < hist for j in range(kt * block_m, min(n, (kt + 1) * block_m)))
                cost = nq - kt if has_history_key else 1
                rows.append((-cost, b, h, kt, offsets[b], n, hist))
    rows.sort()
    it = np.array([(s0, n, h, kt) for (_, b, h, kt, s0, n, _hist) in rows], dtype=np.int32)
    hs = np.array([hist for (*_, hist) in rows], dtype=np.int32)
    return it.reshape(-1, 4), hs


def items_bwd(offsets, heads: int, block_m: int = BLOCK_M) -> np.ndarray:
    """Backward work items: one per (sequence, head, key block kt), which the
    query blocks kt .. nq - 1 see (causal), costing nq - kt; ordered by cost
    descending, then b, h, kt ascending.  int32 (n, 4): (first token, length,
    head, kt)."""
    offsets = [int(x) for x in offsets]
    rows = []
    for b in range(len(offsets) - 1):
        n = offsets[b + 1] - offsets[b]
        nq = (n + block_m - 1) // block_m
        for h in range(heads):
            for kt in range(nq):
                rows.append((-(nq - kt), b, h, kt, offsets[b], n))
    rows.sort()
    out = np.array([(s0, n, h, kt) for (_, b, h, kt, s0, n) in rows], dtype=np.int32)
    return out.reshape(-1, 4)


def items_pairs(offsets, heads: int, block_m: int = BLOCK_M) -> np.ndarray:
    """Pair items: int32 (n, 4) rows (first token, length, head, qp), one per
    two consecutive query blocks of each (sequence, head); cost
    min(2 qp + 2, nq) descending, then b, h, qp ascending."""
    offsets = [int(x) for x in offsets]
    rows = []
    for b in range(len(offsets) - 1):
        n = offsets[b + 1] - offsets[b]
        nq = (n + block_m - 1) // block_m
        for h in range(heads):
            for qp in range((nq + 1) // 2):
                rows.append((-min(2 * qp + 2, nq), b, h, qp, offsets[b], n))
    rows.sort()
    out = np.array([(s0, n, h, qp) for (_, b, h, qp, s0, n) in rows], dtype=np.int32)
    return out.reshape(-1, 4)
