"""Pins of the oracle's backward pass.

HSTU paper Appendix G: the backward recomputes the attention and
accumulates the gradients of the forward definition.  The oracle writes the
chain rule out (hstu_oracle.c).  Pins, each independent of that code:
* central finite differences of the (pinned) forward oracle;
* torch autograd of a dense fp64 formulation (the post's PyTorch
  definition: score matmul, scale, SiLU, tril mask, 1/n, matmul with V);
* linearity: the gradients are linear in dout;
* a one-token sequence's closed form;
* with the bias: torch autograd of the dense definition with the tables
  as parameters and the bias matrix indexed by numpy's float-log2 buckets
  (the tables' gradients included).
"""
import numpy as np
import pytest
import torch

from oracle import reference


def _case(rng, lengths, heads, d, scale=1.0):
    total = int(np.sum(lengths))
    mk = lambda: (scale * rng.standard_normal((total, heads, d))).astype(np.float32)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    return mk(), mk(), mk(), mk(), off


def _loss(q, k, v, dout, off, alpha, inv_n, nt=None, rab=None):
    out = reference.hstu_fwd(q, k, v, off, alpha, inv_n, num_targets=nt, rab=rab)
    return float(np.sum(out * dout.astype(np.float64)))


@pytest.mark.parametrize("targets", [False, True])
def test_finite_differences(targets):
    rng = np.random.default_rng(5 + targets)
    q, k, v, do, off = _case(rng, [6, 0, 9], 2, 4)
    nt = [2, 0, 4] if targets else None
    alpha, inv_n = 0.6, 0.2
    dq, dk, dv = reference.hstu_bwd(q, k, v, do, off, alpha, inv_n, num_targets=nt)
    eps = 1e-3
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0), (3, 1, 2), (5, 0, 3), (6, 1, 1), (14, 0, 0), (10, 1, 3)]:
            xp, xm = x.copy(), x.copy()
            # fp32 inputs: step by a representable amount and use it exactly
            xp[idx] = np.float32(x[idx] + eps)
            xm[idx] = np.float32(x[idx] - eps)
            h = float(xp[idx]) - float(xm[idx])
            args = {"q": q, "k": k, "v": v}
            lp = _loss(*(xp if n == name else args[n] for n in "qkv"), do, off, alpha, inv_n, nt)
            lm = _loss(*(xm if n == name else args[n] for n in "qkv"), do, off, alpha, inv_n, nt)
            fd = (lp - lm) / h
            assert abs(fd - g[idx]) <= 1e-5 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


def _dense_torch(q, k, v, do, off, alpha, inv_n):
    """torch autograd of the dense definition, per sequence, fp64."""
    Q, K, V = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    loss = 0.0
    for b in range(len(off) - 1):
        s0, s1 = int(off[b]), int(off[b + 1])
        if s1 == s0:
            continue
        qb, kb, vb = (x[s0:s1].transpose(0, 1) for x in (Q, K, V))   # (heads, n, d)
        s = alpha * qb @ kb.transpose(1, 2)
        mask = torch.tril(torch.ones(s1 - s0, s1 - s0, dtype=torch.float64))
        p = torch.nn.functional.silu(s) * mask * inv_n
        out = (p @ vb).transpose(0, 1)
        loss = loss + (out * torch.tensor(do[s0:s1], dtype=torch.float64)).sum()
    loss.backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("seed", range(4))
def test_matches_torch_autograd_of_the_dense_definition(seed):
    rng = np.random.default_rng(20 + seed)
    lengths = rng.integers(0, 40, size=4)
    q, k, v, do, off = _case(rng, lengths, 2, 8)
    got = reference.hstu_bwd(q, k, v, do, off, 0.4, 0.05)
    want = _dense_torch(q, k, v, do, off, 0.4, 0.05)
    for g, w_ in zip(got, want):
        assert np.abs(g - w_).max() <= 1e-12 * max(1.0, np.abs(w_).max())


def test_linear_in_dout():
    rng = np.random.default_rng(9)
    q, k, v, _, off = _case(rng, [12, 5], 2, 8)
    # small integers: do + do2 is exact in fp32
    do = rng.integers(-4, 5, size=q.shape).astype(np.float32)
    do2 = rng.integers(-4, 5, size=q.shape).astype(np.float32)
    a = reference.hstu_bwd(q, k, v, do, off, 0.5, 0.1)
    b = reference.hstu_bwd(q, k, v, do2, off, 0.5, 0.1)
    c = reference.hstu_bwd(q, k, v, do + do2, off, 0.5, 0.1)
    for x, y, z in zip(a, b, c):
        assert np.abs(x + y - z).max() <= 1e-12 * max(1.0, np.abs(z).max())


def test_one_token_closed_form():
    rng = np.random.default_rng(10)
    q, k, v, do, off = _case(rng, [1], 1, 4)
    alpha, inv_n = 0.8, 0.5
    dq, dk, dv = reference.hstu_bwd(q, k, v, do, off, alpha, inv_n)
    q0, k0, v0, d0 = (x[0, 0].astype(np.float64) for x in (q, k, v, do))
    x = alpha * q0 @ k0
    sg = 1.0 / (1.0 + np.exp(-x))
    ds = inv_n * sg * (1 + x * (1 - sg)) * (d0 @ v0)
    np.testing.assert_allclose(dv[0, 0], inv_n * x * sg * d0, rtol=1e-13)
    np.testing.assert_allclose(dq[0, 0], alpha * ds * k0, rtol=1e-12)
    np.testing.assert_allclose(dk[0, 0], alpha * ds * q0, rtol=1e-12)


def test_bias_gradients_by_finite_differences():
    # with the relative attention bias the q/k/v gradients still follow the chain rule
    rng = np.random.default_rng(11)
    q, k, v, do, off = _case(rng, [10, 7], 2, 4)
    ts = np.cumsum(rng.integers(0, 5000, size=17)).astype(np.int64)
    pos = (0.3 * rng.standard_normal(8)).astype(np.float32)
    time = (0.3 * rng.standard_normal(16)).astype(np.float32)
    rab = (ts, pos, time)
    dq, dk, dv = reference.hstu_bwd(q, k, v, do, off, 0.6, 0.2, num_targets=[3, 2], rab=rab)
    eps = 1e-3
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 1), (9, 1, 2), (12, 0, 3), (16, 1, 0)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] = np.float32(x[idx] + eps)
            xm[idx] = np.float32(x[idx] - eps)
            h = float(xp[idx]) - float(xm[idx])
            args = {"q": q, "k": k, "v": v}
            lp = _loss(*(xp if n == name else args[n] for n in "qkv"), do, off, 0.6, 0.2, [3, 2], rab)
            lm = _loss(*(xm if n == name else args[n] for n in "qkv"), do, off, 0.6, 0.2, [3, 2], rab)
            assert abs((lp - lm) / h - g[idx]) <= 1e-5 * max(1.0, abs(g[idx])), (name, idx)


def test_sampled_rows_match_the_full_backward():
    rng = np.random.default_rng(12)
    q, k, v, do, off = _case(rng, [50, 3, 90, 1], 2, 8)
    full = reference.hstu_bwd(q, k, v, do, off, 0.5, 0.1)
    rows_t = np.array([0, 29, 49, 50, 52, 53, 100, 142, 143])
    rows_h = np.array([0, 1, 1, 0, 1, 0, 1, 0, 1])
    got = reference.hstu_bwd_rows(q, k, v, do, off, 0.5, 0.1, rows_t, rows_h)
    for g, f in zip(got, full):
        np.testing.assert_allclose(g, f[rows_t, rows_h], rtol=1e-12, atol=1e-15)


def test_sampled_rows_with_the_bias_match_the_full_backward():
    rng = np.random.default_rng(14)
    q, k, v, do, off = _case(rng, [50, 3, 90, 1], 2, 8)
    ts = np.concatenate([np.cumsum(rng.integers(-200, 3000, size=n)) for n in (50, 3, 90, 1)])
    ts = (ts - ts.min()).astype(np.int64)
    pos = (0.4 * rng.standard_normal(7)).astype(np.float32)
    time = (0.4 * rng.standard_normal(20)).astype(np.float32)
    full = reference.hstu_bwd(q, k, v, do, off, 0.5, 0.1, rab=(ts, pos, time))
    plain = reference.hstu_bwd(q, k, v, do, off, 0.5, 0.1)
    rows_t = np.array([0, 29, 49, 50, 52, 53, 100, 142, 143])
    rows_h = np.array([0, 1, 1, 0, 1, 0, 1, 0, 1])
    got = reference.hstu_bwd_rows(q, k, v, do, off, 0.5, 0.1, rows_t, rows_h, rab=(ts, pos, time))
    for g, f, p in zip(got, full, plain):
        np.testing.assert_allclose(g, f[rows_t, rows_h], rtol=1e-12, atol=1e-15)
        # the bias changes the rows (it is not dropped)
        assert np.abs(g - p[rows_t, rows_h]).max() > 1e-3 * np.abs(g).max()


def test_sampled_rows_with_candidates_match_the_full_backward():
    rng = np.random.default_rng(15)
    q, k, v, do, off = _case(rng, [50, 3, 90, 1, 130], 2, 8)
    nt = [20, 3, 0, 1, 129]
    ts = np.concatenate([np.cumsum(rng.integers(0, 3000, size=n)) for n in (50, 3, 90, 1, 130)])
    pos = (0.4 * rng.standard_normal(9)).astype(np.float32)
    time = (0.4 * rng.standard_normal(14)).astype(np.float32)
    rows_t = np.array([0, 29, 30, 49, 50, 52, 53, 142, 143, 144, 200, 273])
    rows_h = np.array([0, 1, 0, 1, 1, 0, 1, 0, 1, 0, 1, 1])
    for rab in (None, (ts.astype(np.int64), pos, time)):
        full = reference.hstu_bwd(q, k, v, do, off, 0.5, 0.1, num_targets=nt, rab=rab)
        causal = reference.hstu_bwd(q, k, v, do, off, 0.5, 0.1, rab=rab)
        got = reference.hstu_bwd_rows(q, k, v, do, off, 0.5, 0.1, rows_t, rows_h, rab=rab,
                                      num_targets=nt)
        for g, f, c in zip(got, full, causal):
            np.testing.assert_allclose(g, f[rows_t, rows_h], rtol=1e-12, atol=1e-15)
        # the mask matters on these rows (candidates see neither each other
        # nor are seen by later candidates)
        assert any(np.abs(g - c[rows_t, rows_h]).max() > 1e-3 * np.abs(g).max()
                   for g, c in zip(got, causal))


def test_bias_table_gradients_by_finite_differences():
    rng = np.random.default_rng(13)
    q, k, v, do, off = _case(rng, [12, 9, 1], 2, 4)
    ts = np.concatenate([np.cumsum(rng.integers(0, 3000, size=n)) for n in (12, 9, 1)]).astype(np.int64)
    pos = (0.3 * rng.standard_normal(6)).astype(np.float32)
    time = (0.3 * rng.standard_normal(12)).astype(np.float32)
    nt = [3, 0, 0]
    got = reference.hstu_bwd(q, k, v, do, off, 0.6, 0.2, num_targets=nt, rab=(ts, pos, time),
                             table_grads=True)
    dpos, dtime = got[3], got[4]
    eps = 1e-3
    for name, tab, g in (("pos", pos, dpos), ("time", time, dtime)):
        for e in range(len(tab)):
            tp, tm = tab.copy(), tab.copy()
            tp[e] = np.float32(tab[e] + eps)
            tm[e] = np.float32(tab[e] - eps)
            h = float(tp[e]) - float(tm[e])
            rp = (ts, tp, time) if name == "pos" else (ts, pos, tp)
            rm = (ts, tm, time) if name == "pos" else (ts, pos, tm)
            fd = (_loss(q, k, v, do, off, 0.6, 0.2, nt, rp) - _loss(q, k, v, do, off, 0.6, 0.2, nt, rm)) / h
            assert abs(fd - g[e]) <= 1e-5 * max(1.0, abs(g[e])), (name, e, fd, g[e])
    # buckets that no kept pair uses get exactly zero
    assert np.count_nonzero(dpos) <= len(pos) and np.all(np.isfinite(dtime))


def _bucket_np(delta, n):
    delta = np.maximum(np.asarray(delta, dtype=np.float64), 0.0)
    return np.minimum(np.floor(np.log2(delta + 1.0)), n - 1).astype(np.int64)


def dense_torch_rab(q, k, v, do, off, ts, pos, time, alpha, inv_n, num_targets=None):
    """torch autograd (fp64) of the dense definition with the bias: the
    tables are leaf tensors, indexed by buckets that numpy computes from
    float log2; candidates (if any) sit at position hist and see the history
    and themselves.  Returns (dq, dk, dv, dpos, dtime)."""
    Q, K, V = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    Pt = torch.tensor(np.asarray(pos, np.float64), requires_grad=True)
    Tt = torch.tensor(np.asarray(time, np.float64), requires_grad=True)
    loss = 0.0
    for b in range(len(off) - 1):
        s0, s1 = int(off[b]), int(off[b + 1])
        n = s1 - s0
        if n == 0:
            continue
        hist = n - (int(num_targets[b]) if num_targets is not None else 0)
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        bp = _bucket_np(np.minimum(i, hist) - np.minimum(j, hist), len(pos))
        t = np.asarray(ts[s0:s1], dtype=np.float64)
        bt = _bucket_np(t[:, None] - t[None, :], len(time))
        mask = torch.tensor(((j <= i) & ((j < hist) | (j == i))).astype(np.float64))
        bias = Pt[torch.tensor(bp)] + Tt[torch.tensor(bt)]
        qb, kb, vb = (x[s0:s1].transpose(0, 1) for x in (Q, K, V))
        s = alpha * qb @ kb.transpose(1, 2) + bias
        p = torch.nn.functional.silu(s) * mask * inv_n
        out = (p @ vb).transpose(0, 1)
        loss = loss + (out * torch.tensor(do[s0:s1], dtype=torch.float64)).sum()
    loss.backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy(), Pt.grad.numpy(), Tt.grad.numpy()


def rab_case(rng, lengths, heads, d, npos, ntime):
    q, k, v, do, off = _case(rng, lengths, heads, d)
    ts = np.concatenate([np.cumsum(rng.integers(-300, 4000, size=int(n))) for n in lengths])
    ts = (ts - (ts.min() if ts.size else 0)).astype(np.int64)
    pos = (0.4 * rng.standard_normal(npos)).astype(np.float32)
    time = (0.4 * rng.standard_normal(ntime)).astype(np.float32)
    return q, k, v, do, off, ts, pos, time


@pytest.mark.parametrize("seed", range(4))
def test_bias_backward_matches_torch_autograd(seed):
    rng = np.random.default_rng(40 + seed)
    lengths = rng.integers(0, 45, size=4)
    nt = [int(rng.integers(0, n + 1)) for n in lengths] if seed % 2 else None
    npos, ntime = int(rng.integers(1, 33)), int(rng.integers(1, 33))
    q, k, v, do, off, ts, pos, time = rab_case(rng, lengths, 2, 8, npos, ntime)
    got = reference.hstu_bwd(q, k, v, do, off, 0.5, 0.07, num_targets=nt, rab=(ts, pos, time),
                             table_grads=True)
    want = dense_torch_rab(q, k, v, do, off, ts, pos, time, 0.5, 0.07, nt)
    for g, w_ in zip(got, want):
        assert np.abs(g - w_).max() <= 1e-12 * max(1.0, np.abs(w_).max())
