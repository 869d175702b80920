"""Pins of the oracle's candidate (M-FALCON) variant.

HSTU paper section 3.4 and Appendix H, Algorithm 1: the last b_m tokens of a
sequence are ranking candidates.  The tril mask is further cleared at
positions (i, j) where both are candidates and i != j, so a candidate sees
the history and itself only.  Appendix H states the identity these pins
rest on: one pass with this mask over history + b_m candidates gives each
candidate exactly the output of a separate causal pass over history + that
one candidate, placed right after the history.

Pins, each independent of the variant's own code path:
* the candidate rows equal the last row of separate causal passes, and the
  history rows equal a causal pass over the history alone.  These use the
  causal oracle, pinned on its own in test_oracle_pins.py;
* no candidates reduces to the causal oracle;
* a sequence of candidates only reduces to a closed form, one term per row;
* brute force with the mask built from the algorithm's steps 4-5;
* the key blocks a query block needs, found by brute force over the mask.
"""
import numpy as np
import pytest
from scipy.special import expit

from oracle import dense, reference, worklist


def _case(rng, lengths, heads, d, scale=1.0):
    total = int(np.sum(lengths))
    mk = lambda: (rng.standard_normal((total, heads, d)) * scale).astype(np.float32)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    return mk(), mk(), mk(), off


def test_no_candidates_is_the_causal_oracle():
    rng = np.random.default_rng(1)
    q, k, v, off = _case(rng, [7, 0, 33, 1, 64], 2, 16)
    a = reference.hstu_fwd(q, k, v, off, 0.3, 0.05)
    b = reference.hstu_fwd(q, k, v, off, 0.3, 0.05, num_targets=[0] * 5)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("hist,bm", [(9, 4), (0, 5), (1, 1), (20, 7), (130, 3)])
def test_candidates_equal_separate_causal_passes(hist, bm):
    rng = np.random.default_rng(100 + hist + bm)
    heads, d, alpha, inv_n = 2, 8, 0.7, 0.01
    q, k, v, off = _case(rng, [hist + bm], heads, d)
    got = reference.hstu_fwd(q, k, v, off, alpha, inv_n, num_targets=[bm])
    for c in range(bm):
        # history followed by candidate c alone: a plain causal pass
        idx = list(range(hist)) + [hist + c]
        sub = reference.hstu_fwd(q[idx], k[idx], v[idx], [0, hist + 1], alpha, inv_n)
        assert np.array_equal(got[hist + c], sub[hist])
    if hist:
        h = reference.hstu_fwd(q[:hist], k[:hist], v[:hist], [0, hist], alpha, inv_n)
        assert np.array_equal(got[:hist], h)


def test_candidates_only_reduce_to_one_term_per_row():
    rng = np.random.default_rng(7)
    q, k, v, off = _case(rng, [6], 3, 8)
    alpha, inv_n = 0.9, 0.25
    got = reference.hstu_fwd(q, k, v, off, alpha, inv_n, num_targets=[6])
    q64, k64, v64 = (t.astype(np.float64) for t in (q, k, v))
    s = alpha * np.einsum("thc,thc->th", q64, k64)
    want = inv_n * (s * expit(s))[..., None] * v64
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-300)


@pytest.mark.parametrize("seed", range(6))
def test_matches_bruteforce_with_the_algorithm_mask(seed):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(0, 40, size=5)
    nt = [int(rng.integers(0, n + 1)) for n in lengths]
    q, k, v, off = _case(rng, lengths, 2, 8)
    got = reference.hstu_fwd(q, k, v, off, 0.4, 0.02, num_targets=nt)
    want = dense.hstu_jagged_bruteforce_targets(q, k, v, off, nt, 0.4, 0.02)
    scale = max(np.abs(want).max(), 1e-300)
    assert np.abs(got - want).max() <= 1e-12 * scale


def test_sampled_rows_match_all_rows():
    rng = np.random.default_rng(3)
    q, k, v, off = _case(rng, [50, 3, 90], 2, 8)
    nt = [20, 3, 0]
    full = reference.hstu_fwd(q, k, v, off, 0.5, 0.1, num_targets=nt)
    rows_t = np.array([0, 29, 30, 49, 50, 52, 53, 142])
    rows_h = np.array([0, 1, 0, 1, 1, 0, 1, 0])
    got = reference.hstu_rows(q, k, v, off, 0.5, 0.1, rows_t, rows_h, num_targets=nt)
    assert np.array_equal(got, full[rows_t, rows_h])


def test_rejects_more_candidates_than_tokens():
    q = np.zeros((4, 1, 8), np.float32)
    with pytest.raises(ValueError):
        reference.hstu_fwd(q, q, q, [0, 4], 1.0, 1.0, num_targets=[5])


def _needed_blocks_bruteforce(n, hist, qt, bm=128):
    """Key blocks holding at least one (i, j) pair the mask keeps, rows of block qt."""
    need = set()
    for i in range(qt * bm, min(n, qt * bm + bm)):
        for j in range(0, i + 1):
            if j < hist or j == i:
                need.add(j // bm)
    return sorted(need)


@pytest.mark.parametrize("n,bm_cand", [(300, 100), (300, 250), (300, 0), (300, 300), (129, 1),
                                       (512, 128), (700, 333), (1, 1)])
def test_worklist_key_blocks_match_bruteforce(n, bm_cand):
    it, hs = worklist.items_targets([0, n], [bm_cand], 1)
    hist = n - bm_cand
    kh = (hist + 127) // 128
    for (s0, length, h, qt), hh in zip(it, hs):
        assert hh == hist and length == n and s0 == 0
        need = _needed_blocks_bruteforce(n, hist, int(qt))
        blocks = list(range(min(int(qt), kh))) + [int(qt)]
        assert need == blocks


def test_worklist_without_candidates_is_the_causal_worklist():
    off = [0, 5, 5, 300, 1000, 1129]
    it, hs = worklist.items_targets(off, [0, 0, 0, 0, 0], 3)
    assert np.array_equal(it, worklist.items(off, 3))
    assert np.array_equal(hs, it[:, 1])


def test_worklist_order_is_cost_descending():
    off = [0, 300, 1000]
    it, hs = worklist.items_targets(off, [250, 100], 2)
    kh = (hs + 127) // 128
    cost = np.minimum(it[:, 3], kh) + 1
    assert np.all(np.diff(cost) <= 0)
