"""Padded-dense brute force of the HSTU formula (numpy float64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

This evaluates the post's PyTorch definition (ai6s.net "HSTU fused operator"
post, section 1) on padded head-major tensors (b, heads, s, d) with an
explicit (b, heads, s, s) mask, in the definition's order of operations:
scores = Q K^T; scores * alpha; silu; multiply by mask / n; result @ V.
The mask is the decoder tril including the diagonal (section 3.1), and
padding is the dense layout that section 4.1 describes.  Padded query rows
are discarded; padded keys are masked out because they sit above the
diagonal of every valid row.
"""
from __future__ import annotations

import numpy as np


def _sigmoid(x: np.ndarray) -> np.ndarray:
    # numerically safe logistic: exp of a non-positive argument only
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def jagged_to_padded(x: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """(total, heads, d) jagged -> (b, heads, max_s, d) zero padded, head-major."""
    b = len(offsets) - 1
    lens = np.diff(offsets)
    s = int(lens.max()) if b else 0
    total, heads, d = x.shape
    out = np.zeros((b, heads, s, d), dtype=np.float64)
    for i in range(b):
        seg = x[offsets[i]:offsets[i + 1]]  # (n_i, heads, d)
        out[i, :, :lens[i], :] = np.transpose(seg, (1, 0, 2))
    return out


def padded_to_jagged(y: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    b, heads, s, d = y.shape
    total = int(offsets[-1])
    out = np.zeros((total, heads, d), dtype=np.float64)
    for i in range(b):
        n = offsets[i + 1] - offsets[i]
        out[offsets[i]:offsets[i + 1]] = np.transpose(y[i, :, :n, :], (1, 0, 2))
    return out


def hstu_dense(Q: np.ndarray, K: np.ndarray, V: np.ndarray, mask: np.ndarray, alpha: float,
               n: float) -> np.ndarray:
    """Head-major dense HSTU: Q, K, V (b, heads, s, d); mask (b, heads, s, s)."""
    scores = np.matmul(Q, np.swapaxes(K, -1, -2))           # (b, heads, s, s)
    scores = scores * alpha
    scores = scores * _sigmoid(scores)                       # silu
    scores = scores * (mask / n)
    return np.matmul(scores, V)                              # (b, heads, s, d)


def causal_mask(b: int, heads: int, s: int) -> np.ndarray:
    return np.broadcast_to(np.tril(np.ones((s, s), dtype=np.float64)), (b, heads, s, s)).copy()


def hstu_jagged_bruteforce(q, k, v, offsets, alpha: float, inv_n: float) -> np.ndarray:
    """Jagged in, jagged out, via the padded-dense definition.  Tiny inputs only."""
    offsets = np.asarray(offsets, dtype=np.int64)
    q64, k64, v64 = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    Q, K, V = (jagged_to_padded(t, offsets) for t in (q64, k64, v64))
    b, heads, s, _ = Q.shape
    y = hstu_dense(Q, K, V, causal_mask(b, heads, s), alpha, 1.0 / inv_n)
    return padded_to_jagged(y, offsets)


def candidate_mask(lengths, num_targets, heads: int, s: int) -> np.ndarray:
    """The M-FALCON mask (HSTU paper Appendix H, Algorithm 1 steps 4-5) per
    sequence: the tril matrix, then position (i, j) cleared wherever both i
    and j are candidate positions (>= hist = n - num_targets) and i != j."""
    b = len(lengths)
    m = np.zeros((b, heads, s, s), dtype=np.float64)
    for i in range(b):
        hist = int(lengths[i]) - int(num_targets[i])
        L = np.tril(np.ones((s, s), dtype=np.float64))      # step 4
        for r in range(hist, s):                             # step 5
            for c in range(hist, s):
                if r != c:
                    L[r, c] = 0.0
        m[i] = L
    return m


def hstu_jagged_bruteforce_targets(q, k, v, offsets, num_targets, alpha: float,
                                   inv_n: float) -> np.ndarray:
    """As hstu_jagged_bruteforce, with the M-FALCON mask.  Tiny inputs only."""
    offsets = np.asarray(offsets, dtype=np.int64)
    q64, k64, v64 = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    Q, K, V = (jagged_to_padded(t, offsets) for t in (q64, k64, v64))
    b, heads, s, _ = Q.shape
    mask = candidate_mask(np.diff(offsets), num_targets, heads, s)
    y = hstu_dense(Q, K, V, mask, alpha, 1.0 / inv_n)
    return padded_to_jagged(y, offsets)
