"""Pins of the oracle's relative attention bias rab_{p,t}.

HSTU paper section 3: rab_{p,t} is a relative attention bias that merges
position p and time t, added inside the attention's nonlinearity.  Section
3.4: M-FALCON modifies it for candidates.  Appendix G: its construction is
fused into the attention operator.  The construction is lost in
extraction; the reading (hstu_oracle.c) is a pair of bucketed tables:

    silu(alpha q_i.k_j + pos[min(floor(log2(dp+1)), P-1)] + time[min(floor(log2(dt+1)), B-1)])

dp = p(i) - p(j) with every candidate at position hist, dt = max(ts_i - ts_j, 0).

Pins, each independent of the oracle's own code:
* the bucket function against numpy's floating-point log2 over a range of
  deltas that includes every power-of-two edge;
* zero tables reduce to the causal oracle;
* brute force: the post's dense definition with a bias matrix built by
  numpy from floating-point log2;
* row 0 of a sequence has the closed form silu(alpha q0.k0 + pos[0] + time[0]);
* Appendix H's identity with the bias: one pass with candidates equals
  separate causal passes over history + one candidate.
"""
import numpy as np
import pytest
from scipy.special import expit

from oracle import reference


def _bucket_np(delta, n):
    delta = np.maximum(np.asarray(delta, dtype=np.float64), 0.0)
    return np.minimum(np.floor(np.log2(delta + 1.0)), n - 1).astype(np.int64)


def test_bucket_against_float_log2():
    deltas = [0, 1, 2, 3, 4, 5, 6, 7, 8, 15, 16, 17, 1023, 1024, 1025, -1, -5, -(2 ** 40)]
    deltas += [2 ** k - 1 for k in range(1, 32)] + [2 ** k for k in range(1, 32)]
    for n in (1, 2, 8, 32):
        for dlt in deltas:
            assert reference.rab_bucket(dlt, n) == int(_bucket_np(dlt, n)), (dlt, n)


def _case(rng, lengths, heads, d):
    total = int(np.sum(lengths))
    mk = lambda: rng.standard_normal((total, heads, d)).astype(np.float32)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    # timestamps: increasing within a sequence with log-normal gaps, plus a
    # few steps backwards to exercise the clamp at dt = 0
    ts = np.zeros(total, dtype=np.int64)
    for b in range(len(lengths)):
        gaps = np.exp(rng.normal(4.0, 3.0, size=int(lengths[b]))).astype(np.int64)
        gaps[rng.random(int(lengths[b])) < 0.1] *= -1
        ts[off[b]:off[b + 1]] = 1_000_000 + np.cumsum(gaps)
    return mk(), mk(), mk(), off, ts


def _tables(rng, npos, ntime, scale=0.5):
    return ((scale * rng.standard_normal(npos)).astype(np.float32),
            (scale * rng.standard_normal(ntime)).astype(np.float32))


def test_zero_tables_are_the_causal_oracle():
    rng = np.random.default_rng(1)
    q, k, v, off, ts = _case(rng, [7, 0, 33, 1, 64], 2, 16)
    a = reference.hstu_fwd(q, k, v, off, 0.3, 0.05)
    b = reference.hstu_fwd(q, k, v, off, 0.3, 0.05,
                           rab=(ts, np.zeros(8, np.float32), np.zeros(32, np.float32)))
    assert np.array_equal(a, b)


def _bruteforce(q, k, v, off, ts, pos, time, alpha, inv_n, num_targets=None):
    """The post's dense definition on each sequence, with the bias matrix
    built by numpy (float log2 buckets), the tril mask cleared at
    candidate-candidate pairs (Appendix H)."""
    total, heads, d = q.shape
    out = np.zeros((total, heads, d))
    for b in range(len(off) - 1):
        s0, s1 = int(off[b]), int(off[b + 1])
        n = s1 - s0
        if n == 0:
            continue
        hist = n - (int(num_targets[b]) if num_targets is not None else 0)
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        pi, pj = np.minimum(i, hist), np.minimum(j, hist)
        t = ts[s0:s1].astype(np.float64)
        bias = (pos.astype(np.float64)[_bucket_np(pi - pj, len(pos))]
                + time.astype(np.float64)[_bucket_np(t[:, None] - t[None, :], len(time))])
        mask = (j <= i) & ((j < hist) | (j == i))
        for h in range(heads):
            s = alpha * (q[s0:s1, h].astype(np.float64) @ k[s0:s1, h].astype(np.float64).T) + bias
            p = s * expit(s) * mask
            out[s0:s1, h] = inv_n * (p @ v[s0:s1, h].astype(np.float64))
    return out


@pytest.mark.parametrize("seed", range(6))
def test_matches_bruteforce(seed):
    rng = np.random.default_rng(10 + seed)
    lengths = rng.integers(0, 50, size=4)
    nt = [int(rng.integers(0, n + 1)) for n in lengths] if seed % 2 else None
    q, k, v, off, ts = _case(rng, lengths, 2, 8)
    pos, time = _tables(rng, int(rng.integers(1, 33)), int(rng.integers(1, 33)))
    got = reference.hstu_fwd(q, k, v, off, 0.4, 0.02, num_targets=nt, rab=(ts, pos, time))
    want = _bruteforce(q, k, v, off, ts, pos, time, 0.4, 0.02, nt)
    scale = max(np.abs(want).max(), 1e-300)
    assert np.abs(got - want).max() <= 1e-12 * scale


def test_first_row_closed_form():
    rng = np.random.default_rng(3)
    q, k, v, off, ts = _case(rng, [5, 9], 3, 8)
    pos, time = _tables(rng, 16, 16)
    got = reference.hstu_fwd(q, k, v, off, 0.7, 0.25, rab=(ts, pos, time))
    for t in off[:-1]:
        s = 0.7 * np.einsum("hc,hc->h", q[t].astype(np.float64), k[t].astype(np.float64))
        s = s + float(pos[0]) + float(time[0])
        want = 0.25 * (s * expit(s))[:, None] * v[t].astype(np.float64)
        np.testing.assert_allclose(got[t], want, rtol=1e-13)


@pytest.mark.parametrize("hist,bm", [(9, 4), (0, 3), (20, 5), (130, 2)])
def test_candidates_equal_separate_causal_passes_with_bias(hist, bm):
    rng = np.random.default_rng(100 + hist)
    q, k, v, off, ts = _case(rng, [hist + bm], 2, 8)
    pos, time = _tables(rng, 32, 32)
    got = reference.hstu_fwd(q, k, v, off, 0.6, 0.1, num_targets=[bm], rab=(ts, pos, time))
    for c in range(bm):
        idx = list(range(hist)) + [hist + c]
        sub = reference.hstu_fwd(q[idx], k[idx], v[idx], [0, hist + 1], 0.6, 0.1,
                                 rab=(ts[idx], pos, time))
        assert np.array_equal(got[hist + c], sub[hist])


def test_sampled_rows_match_all_rows():
    rng = np.random.default_rng(4)
    q, k, v, off, ts = _case(rng, [50, 3, 90], 2, 8)
    pos, time = _tables(rng, 12, 20)
    nt = [20, 1, 0]
    full = reference.hstu_fwd(q, k, v, off, 0.5, 0.1, num_targets=nt, rab=(ts, pos, time))
    rows_t = np.array([0, 29, 30, 49, 50, 52, 53, 142])
    rows_h = np.array([0, 1, 0, 1, 1, 0, 1, 0])
    got = reference.hstu_rows(q, k, v, off, 0.5, 0.1, rows_t, rows_h, num_targets=nt,
                              rab=(ts, pos, time))
    assert np.array_equal(got, full[rows_t, rows_h])


def test_rejects_bad_tables():
    q = np.zeros((4, 1, 8), np.float32)
    with pytest.raises(ValueError):
        reference.hstu_fwd(q, q, q, [0, 4], 1.0, 1.0, rab=(np.zeros(3), [0.0], [0.0]))
    with pytest.raises(ValueError):
        reference.hstu_fwd(q, q, q, [0, 4], 1.0, 1.0, rab=(np.zeros(4), [], [0.0]))
