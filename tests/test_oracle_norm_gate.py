"""Pins of the oracle's output stage, Norm(A V) (.) U.

HSTU paper section 3: each layer's spatial aggregation is followed by a
pointwise transformation.  Section 3.1 requires a layer norm after the
pointwise pooling, and the feature-interaction paragraph writes the term as
Norm(A(X) V(X)) (.) U(X).  The equations are lost in extraction.  The
reading taken is a standard layer norm over each token's heads * d outputs,
with affine gamma and beta, times U elementwise.

Pins, each independent of the oracle's own code:
* torch's layer_norm (fp64), a library routine, times u;
* the closed form of a two-wide row with eps = 0: the normalised pair is
  (+1, -1) or (-1, +1);
* invariance to a positive scale and a shift of the row (eps = 0), so that
  inv_n cancels from the whole fused op;
* the composition with the padded-dense brute force of the attention;
* the candidate identity of Appendix H carries over token by token.
"""
import numpy as np
import pytest
import torch

from oracle import dense, reference


def _ln_torch(x, u, g, b, eps):
    rows, heads, d = x.shape
    t = torch.nn.functional.layer_norm(torch.tensor(x.reshape(rows, heads * d), dtype=torch.float64),
                                       (heads * d,), torch.tensor(g, dtype=torch.float64),
                                       torch.tensor(b, dtype=torch.float64), eps)
    return t.numpy().reshape(rows, heads, d) * u.astype(np.float64)


def _params(rng, heads, d):
    g = (1.0 + 0.3 * rng.standard_normal(heads * d)).astype(np.float32)
    b = (0.3 * rng.standard_normal(heads * d)).astype(np.float32)
    return g, b


@pytest.mark.parametrize("rows,heads,d,eps", [(7, 2, 8, 1e-5), (3, 4, 16, 0.0), (5, 1, 1, 1e-6),
                                              (4, 3, 5, 0.5), (0, 2, 4, 1e-5)])
def test_matches_torch_layer_norm_times_u(rows, heads, d, eps):
    rng = np.random.default_rng(rows * 100 + heads * 10 + d)
    x = rng.standard_normal((rows, heads, d)) * 3.0 + 0.7
    u = rng.standard_normal((rows, heads, d)).astype(np.float32)
    g, b = _params(rng, heads, d)
    got = reference.norm_gate(x, u, g, b, eps)
    want = _ln_torch(x, u, g, b, eps)
    assert got.shape == want.shape
    if rows:
        assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


def test_two_wide_row_closed_form():
    # width 2, eps = 0: (x - mean) / std is +-1 whenever the two differ
    x = np.array([[[3.0], [-1.5]], [[-2.0], [7.0]], [[1e-3], [0.0]]])
    u = np.array([[[2.0], [0.5]], [[1.0], [-1.0]], [[4.0], [3.0]]], dtype=np.float32)
    g = np.array([1.5, -0.5], dtype=np.float32)
    b = np.array([0.25, 2.0], dtype=np.float32)
    got = reference.norm_gate(x, u, g, b, 0.0)
    sign = np.sign(x[:, 0, 0] - x[:, 1, 0])
    want = np.stack([(sign * 1.5 + 0.25) * u[:, 0, 0], (-sign * -0.5 + 2.0) * u[:, 1, 0]], axis=1)
    np.testing.assert_allclose(got[:, :, 0], want, rtol=1e-12)


def test_width_one_keeps_only_beta():
    x = np.array([[[5.0]], [[-3.0]]])
    u = np.array([[[2.0]], [[-1.0]]], dtype=np.float32)
    got = reference.norm_gate(x, u, np.array([9.0], np.float32), np.array([0.5], np.float32), 1e-5)
    np.testing.assert_array_equal(got[:, 0, 0], [1.0, -0.5])


def test_scale_and_shift_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 2, 8))
    u = rng.standard_normal((6, 2, 8)).astype(np.float32)
    g, b = _params(rng, 2, 8)
    a = reference.norm_gate(x, u, g, b, 0.0)
    c = reference.norm_gate(x * 37.5 - 4.25, u, g, b, 0.0)
    assert np.abs(a - c).max() <= 1e-12 * np.abs(a).max()


def test_standardised_rows():
    # gamma = 1, beta = 0, u = 1: each row has mean 0 and mean square var / (var + eps)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, 4, 8)) * 0.1
    ones = np.ones((5, 4, 8), np.float32)
    eps = 1e-3
    y = reference.norm_gate(x, ones, np.ones(32, np.float32), np.zeros(32, np.float32), eps)
    rows = y.reshape(5, 32)
    var = x.reshape(5, 32).var(axis=1)
    np.testing.assert_allclose(rows.mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose((rows ** 2).mean(axis=1), var / (var + eps), rtol=1e-12)


def _case(rng, lengths, heads, d):
    total = int(np.sum(lengths))
    mk = lambda: rng.standard_normal((total, heads, d)).astype(np.float32)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    return mk(), mk(), mk(), off


@pytest.mark.parametrize("seed", range(4))
def test_fused_op_equals_layer_norm_of_the_bruteforce(seed):
    rng = np.random.default_rng(40 + seed)
    lengths = rng.integers(0, 30, size=4)
    heads, d = 2, 8
    q, k, v, off = _case(rng, lengths, heads, d)
    u = rng.standard_normal(q.shape).astype(np.float32)
    g, b = _params(rng, heads, d)
    got = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, 1e-5, off, 0.4, 0.05)
    attn = dense.hstu_jagged_bruteforce(q, k, v, off, 0.4, 0.05)
    want = _ln_torch(attn, u, g, b, 1e-5)
    assert np.abs(got - want).max() <= 1e-10 * max(1.0, np.abs(want).max())


def test_inv_n_cancels_without_eps():
    rng = np.random.default_rng(9)
    q, k, v, off = _case(rng, [17, 1, 40], 2, 8)
    u = rng.standard_normal(q.shape).astype(np.float32)
    g, b = _params(rng, 2, 8)
    a = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, 0.0, off, 0.5, 1.0)
    c = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, 0.0, off, 0.5, 1.0 / 4096)
    assert np.abs(a - c).max() <= 1e-11 * np.abs(a).max()


def test_sampled_tokens_match_all_tokens():
    rng = np.random.default_rng(10)
    q, k, v, off = _case(rng, [50, 3, 90], 3, 8)
    u = rng.standard_normal(q.shape).astype(np.float32)
    g, b = _params(rng, 3, 8)
    full = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, 1e-5, off, 0.5, 0.1, num_targets=[20, 1, 0])
    rows = np.array([0, 29, 30, 49, 50, 52, 53, 142])
    got = reference.hstu_rows_norm_gate(q, k, v, u, g, b, 1e-5, off, 0.5, 0.1, rows,
                                        num_targets=[20, 1, 0])
    assert np.array_equal(got, full[rows])


def test_candidate_identity_carries_over():
    # the norm acts per token, so a candidate's output still equals the last
    # row of a separate causal pass over history + that candidate
    rng = np.random.default_rng(11)
    hist, bm, heads, d = 13, 4, 2, 8
    q, k, v, off = _case(rng, [hist + bm], heads, d)
    u = rng.standard_normal(q.shape).astype(np.float32)
    g, b = _params(rng, heads, d)
    got = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, 1e-5, off, 0.7, 0.1, num_targets=[bm])
    for c in range(bm):
        idx = list(range(hist)) + [hist + c]
        sub = reference.hstu_fwd_norm_gate(q[idx], k[idx], v[idx], u[idx], g, b, 1e-5,
                                           [0, hist + 1], 0.7, 0.1)
        assert np.array_equal(got[hist + c], sub[hist])


def test_rejects_bad_arguments():
    x = np.zeros((2, 2, 4))
    u = np.zeros((2, 2, 4), np.float32)
    g = np.ones(8, np.float32)
    with pytest.raises(ValueError):
        reference.norm_gate(x, u, g, g, -1.0)
    with pytest.raises(ValueError):
        reference.norm_gate(x, u, g[:4], g, 1e-5)

