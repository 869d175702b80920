"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a closed form, a limit, a library routine,
brute force on tiny inputs, an invariant of the formula, or hand-worked
values, so that a plausible slip in the oracle fails at least one of them:

* a dropped diagonal term or an off-by-one in the key range: row-0 closed
  form, brute force, constant-V prefix sums;
* a wrong sign inside silu: the large-alpha ReLU limit, library sigmoid;
* alpha applied as a divisor or misplaced: odd-part identity, brute force;
* transposed operands (q.v or k.v): brute force with distinct q, k, v;
* wrong head or sequence indexing: brute force, head permutation,
  cross-sequence isolation, empty sequences.

The formula is the ai6s.net "HSTU fused operator" post, section 1 (HSTU
formula and PyTorch definition), section 3.2 (tril block mask including the
diagonal), section 4.2 (jagged values + offsets); HSTU paper section 3.1
(pointwise aggregated attention, no softmax).
"""
import math

import numpy as np
import pytest
from scipy.special import expit

from oracle import dense, reference, worklist
from hstu_jagged_attention_gb300 import workloads

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_case(rng, lengths, heads, d, scale=1.0, integer=False):
    total = int(np.sum(lengths))
    if integer:
        mk = lambda: rng.integers(-3, 4, size=(total, heads, d)).astype(np.float32)
    else:
        mk = lambda: (rng.standard_normal((total, heads, d)) * scale).astype(np.float32)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    return mk(), mk(), mk(), off


# --------------------------------------------------------------------- silu
@pytest.mark.parametrize("x", [-800.0, -40.0, -5.5, -1.0, -1e-8, 0.0, 1e-8, 0.5, 1.0, 3.0, 40.0, 800.0])
def test_silu_matches_library_sigmoid(x):
    # silu(x) = x * sigmoid(x); scipy's expit is an independent logistic routine.
    assert reference.silu(x) == pytest.approx(x * expit(x), rel=1e-15, abs=1e-300)


def test_silu_special_values():
    assert reference.silu(0.0) == 0.0
    assert reference.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    # minimum of silu is at the root of 1 + x + e^x = 0 ... i.e. x ~= -1.2784645, value ~= -0.2784645
    xs = np.linspace(-3, 0, 30001)
    vals = np.array([reference.silu(x) for x in xs])
    assert xs[vals.argmin()] == pytest.approx(-1.2784645, abs=2e-4)
    assert vals.min() == pytest.approx(-0.2784645, abs=1e-6)


def test_dense_sigmoid_matches_library():
    x = np.linspace(-50, 50, 1001)
    np.testing.assert_allclose(dense._sigmoid(x), expit(x), rtol=1e-14, atol=0)


# ----------------------------------------------------------- closed forms
def test_row0_closed_form():
    rng = np.random.default_rng(7)
    q, k, v, off = _rand_case(rng, [5, 1, 9, 3], heads=3, d=16)
    alpha, inv_n = 0.37, 0.11
    out = reference.hstu_fwd(q, k, v, off, alpha, inv_n)
    for b in range(len(off) - 1):
        t = off[b]
        for h in range(3):
            s = float(np.dot(q[t, h].astype(np.float64), k[t, h].astype(np.float64)))
            expect = inv_n * (alpha * s) * expit(alpha * s) * v[t, h].astype(np.float64)
            np.testing.assert_allclose(out[t, h], expect, rtol=1e-13, atol=1e-300)


def test_alpha_zero_gives_exact_zero():
    rng = np.random.default_rng(1)
    q, k, v, off = _rand_case(rng, [13, 40, 2], heads=2, d=8)
    out = reference.hstu_fwd(q, k, v, off, 0.0, 0.5)
    assert np.all(out == 0.0)


def test_zero_keys_give_exact_zero():
    rng = np.random.default_rng(2)
    q, k, v, off = _rand_case(rng, [13, 40, 2], heads=2, d=8)
    k[:] = 0
    out = reference.hstu_fwd(q, k, v, off, 0.3, 0.5)
    assert np.all(out == 0.0)


def test_constant_v_is_prefix_sum_of_scores():
    # with v == 1 every output coordinate is inv_n * sum_{j<=i} silu(alpha s_ij);
    # computed here as a cumulative sum over a full score matrix (numpy + expit).
    rng = np.random.default_rng(3)
    q, k, v, off = _rand_case(rng, [37], heads=1, d=8)
    v[:] = 1.0
    alpha, inv_n = 0.6, 0.125
    out = reference.hstu_fwd(q, k, v, off, alpha, inv_n)
    S = alpha * (q[:, 0].astype(np.float64) @ k[:, 0].astype(np.float64).T)
    P = S * expit(S)
    for i in range(37):
        ref = inv_n * np.cumsum(P[i])[i]
        np.testing.assert_allclose(out[i, 0], np.full(8, ref), rtol=1e-12)


def test_large_alpha_limit_is_relu_attention():
    # silu(a x)/a -> relu(x) as a -> inf.  Integer q, k make every score an integer,
    # so |score| >= 1 or score == 0 and the limit is reached to machine precision.
    rng = np.random.default_rng(4)
    q, k, v, off = _rand_case(rng, [19, 6], heads=2, d=4, integer=True)
    a = 200.0
    out = reference.hstu_fwd(q, k, v, off, a, 1.0) / a
    for b in range(2):
        s0, s1 = off[b], off[b + 1]
        for h in range(2):
            S = q[s0:s1, h].astype(np.float64) @ k[s0:s1, h].astype(np.float64).T
            ref = np.tril(np.maximum(S, 0.0)) @ v[s0:s1, h].astype(np.float64)
            np.testing.assert_allclose(out[s0:s1, h], ref, rtol=1e-12, atol=1e-12)


def test_odd_part_is_linear_causal_attention():
    # silu(x) - silu(-x) = x  =>  out(q) - out(-q) = alpha inv_n tril(q k^T) v.
    rng = np.random.default_rng(5)
    q, k, v, off = _rand_case(rng, [23, 11], heads=2, d=8)
    alpha, inv_n = 0.45, 0.2
    diff = reference.hstu_fwd(q, k, v, off, alpha, inv_n) - reference.hstu_fwd(-q, k, v, off, alpha, inv_n)
    for b in range(2):
        s0, s1 = off[b], off[b + 1]
        for h in range(2):
            S = q[s0:s1, h].astype(np.float64) @ k[s0:s1, h].astype(np.float64).T
            ref = alpha * inv_n * (np.tril(S) @ v[s0:s1, h].astype(np.float64))
            np.testing.assert_allclose(diff[s0:s1, h], ref, rtol=1e-10, atol=1e-12)


# -------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed", range(6))
def test_matches_padded_dense_bruteforce(seed):
    rng = np.random.default_rng(100 + seed)
    nb = int(rng.integers(1, 6))
    lengths = rng.integers(0, 71, size=nb)
    heads = int(rng.integers(1, 4))
    d = int(rng.choice([1, 3, 8, 16]))
    q, k, v, off = _rand_case(rng, lengths, heads, d)
    alpha = float(rng.uniform(0.05, 1.5))
    inv_n = float(1.0 / rng.integers(1, 100))
    got = reference.hstu_fwd(q, k, v, off, alpha, inv_n)
    ref = dense.hstu_jagged_bruteforce(q, k, v, off, alpha, inv_n)
    scale = max(np.abs(ref).max(), 1e-300)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13 * scale)


def test_tiny_workload_matches_bruteforce():
    w = workloads.workload("tiny")
    q, k, v = workloads.draw_qkv(w)
    got = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n)
    ref = dense.hstu_jagged_bruteforce(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                       w.offsets, w.alpha, w.inv_n)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_bruteforce_dense_mask_is_tril_with_diagonal():
    m = dense.causal_mask(1, 1, 4)[0, 0]
    assert m.tolist() == [[1, 0, 0, 0], [1, 1, 0, 0], [1, 1, 1, 0], [1, 1, 1, 1]]


# --------------------------------------------------------------- invariants
def test_causality_future_keys_values_do_not_matter():
    rng = np.random.default_rng(8)
    q, k, v, off = _rand_case(rng, [50], heads=2, d=8)
    base = reference.hstu_fwd(q, k, v, off, 0.3, 0.1)
    for i in (0, 17, 48):
        k2, v2 = k.copy(), v.copy()
        k2[i + 1:] = rng.standard_normal(k2[i + 1:].shape) * 5
        v2[i + 1:] = rng.standard_normal(v2[i + 1:].shape) * 5
        out = reference.hstu_fwd(q, k2, v2, off, 0.3, 0.1)
        assert np.array_equal(out[: i + 1], base[: i + 1])
        assert not np.array_equal(out[i + 1:], base[i + 1:])


def test_sequences_are_isolated():
    rng = np.random.default_rng(9)
    q, k, v, off = _rand_case(rng, [10, 20, 5], heads=2, d=8)
    base = reference.hstu_fwd(q, k, v, off, 0.3, 0.1)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    sl = slice(off[1], off[2])
    q2[sl] += 1
    k2[sl] -= 2
    v2[sl] *= 3
    out = reference.hstu_fwd(q2, k2, v2, off, 0.3, 0.1)
    assert np.array_equal(out[: off[1]], base[: off[1]])
    assert np.array_equal(out[off[2]:], base[off[2]:])


def test_empty_sequences_produce_no_rows_and_change_nothing():
    rng = np.random.default_rng(10)
    lengths = [6, 9, 4]
    q, k, v, off = _rand_case(rng, lengths, heads=2, d=8)
    base = reference.hstu_fwd(q, k, v, off, 0.3, 0.1)
    off_e = np.array([0, 0, 6, 6, 6, 15, 19, 19], dtype=np.int64)  # empties interleaved
    out = reference.hstu_fwd(q, k, v, off_e, 0.3, 0.1)
    assert out.shape == base.shape
    assert np.array_equal(out, base)
    empty = reference.hstu_fwd(q[:0], k[:0], v[:0], np.zeros(4, np.int64), 0.3, 0.1)
    assert empty.shape == (0, 2, 8)


def test_head_permutation_commutes():
    rng = np.random.default_rng(11)
    q, k, v, off = _rand_case(rng, [12, 7], heads=4, d=8)
    perm = np.array([2, 0, 3, 1])
    base = reference.hstu_fwd(q, k, v, off, 0.3, 0.1)
    out = reference.hstu_fwd(q[:, perm], k[:, perm], v[:, perm], off, 0.3, 0.1)
    assert np.array_equal(out, base[:, perm])


def test_linear_in_v_and_inv_n():
    rng = np.random.default_rng(12)
    q, k, v, off = _rand_case(rng, [15, 8], heads=2, d=8)
    v2 = (rng.standard_normal(v.shape)).astype(np.float32)
    a = reference.hstu_fwd(q, k, v, off, 0.3, 0.1)
    b = reference.hstu_fwd(q, k, v2, off, 0.3, 0.1)
    c = reference.hstu_fwd(q, k, v + v2, off, 0.3, 0.1)  # v + v2 is exact? not always: allow rounding
    np.testing.assert_allclose(c, a + b, rtol=1e-6, atol=1e-6)
    d2 = reference.hstu_fwd(q, k, v, off, 0.3, 0.4)
    np.testing.assert_allclose(d2, 4 * a, rtol=1e-14)


def test_sampled_rows_equal_full_rows():
    rng = np.random.default_rng(13)
    q, k, v, off = _rand_case(rng, [30, 0, 45, 1], heads=3, d=8)
    full = reference.hstu_fwd(q, k, v, off, 0.3, 0.1)
    rt = np.array([0, 29, 30, 74, 75, 44, 5])
    rh = np.array([0, 2, 1, 1, 0, 2, 1])
    rows = reference.hstu_rows(q, k, v, off, 0.3, 0.1, rt, rh)
    assert np.array_equal(rows, full[rt, rh])
    # a token outside every sequence yields NaN, not a value
    bad = reference.hstu_rows(q, k, v, off, 0.3, 0.1, np.array([76]), np.array([0]))
    assert np.isnan(bad).all()


def test_rejects_bad_offsets():
    q = np.zeros((4, 1, 2), np.float32)
    with pytest.raises(ValueError):
        reference.hstu_fwd(q, q, q, np.array([0, 3, 2, 4]), 1.0, 1.0)


# ---------------------------------------------------------------- work list
def _read_worklist_cases():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "worklist_hand_cases.txt")
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case"):
            kv = dict(p.split("=") for p in line.split()[1:])
            cur = ([int(x) for x in kv["offsets"].split(",")], int(kv["heads"]), [])
            cases.append(cur)
        else:
            cur[2].append([int(x) for x in line.split()])
    return cases


def test_worklist_hand_cases():
    cases = _read_worklist_cases()
    assert len(cases) == 4
    for offsets, heads, expect in cases:
        got = worklist.items(offsets, heads)
        assert got.tolist() == expect


@pytest.mark.parametrize("name", workloads.WORKLOAD_NAMES)
def test_worklist_invariants(name):
    w = workloads.workload(name)
    it = worklist.items(w.offsets, w.heads)
    tiles = (w.lengths + 127) // 128
    assert len(it) == w.heads * int(tiles.sum())
    cost = it[:, 3] + 1
    assert np.all(np.diff(cost) <= 0)  # longest first
    # each (seq, head, qt) once, qt within the sequence's block range
    keys = {(int(a), int(c), int(d_)) for a, _, c, d_ in it}
    assert len(keys) == len(it)
    assert np.all(it[:, 3] * 128 < it[:, 1])


# --------------------------------------------------- the page's memory figures
def test_page_memory_figures_reading():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "page_memory_figures.txt")
    fig = {}
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            key, val = line.split()
            fig[key] = float(val)
    b, n, s, d = (int(fig[x]) for x in ("batch", "heads", "s", "d"))
    G = 2.0 ** 30
    qkvo = 4 * b * n * s * d * 2
    mask = b * n * s * s * 2
    assert mask / G == fig["mask_GiB"]
    assert (qkvo + 2 * mask) / G == fig["small_ops_GiB"]
    assert (qkvo + mask) / G == fig["fused_GiB"]
    assert qkvo / G == fig["fused_builtin_mask_GiB"]
