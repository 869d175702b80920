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
