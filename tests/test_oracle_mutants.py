"""The oracle pins must catch plausible mistakes.

Each case copies the C oracle into a temporary directory, plants one
mistake in the copy, builds it, and checks that a pin from
``test_oracle_pins.py`` now fails.  The committed oracle is untouched.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
from scipy.special import expit

from oracle import build as oracle_build
from oracle import dense

MUTANTS = {
    "silu_sign": ("x / (1.0 + exp(-x))", "x / (1.0 + exp(x))"),
    "drop_diagonal": ("return j <= i && (j < hist || j == i);", "return j < i && (j < hist || j == i);"),
    "alpha_divides": ("hstu_oracle_silu(alpha * dot + bias)", "hstu_oracle_silu(dot / alpha + bias)"),
    "q_dot_v": ("dot += (double)qr[c] * (double)kr[c]", "dot += (double)qr[c] * (double)vr[c]"),
    "inv_n_missing": ("out_row[c] = inv_n * acc[c]", "out_row[c] = acc[c]"),
    "wrong_head_stride": ("(s * heads + h) * (int64_t)d;\n        const float* vr",
                          "(s * heads + 0) * (int64_t)d;\n        const float* vr"),
}


def _build_mutant(tmp_path, name):
    src = open(oracle_build.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", str(lib), str(path),
                    "-lm", "-lpthread"], check=True)
    L = ctypes.CDLL(str(lib))
    f, dptr, i64 = (ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                    ctypes.POINTER(ctypes.c_int64))
    L.hstu_oracle_fwd_f64.argtypes = [f, f, f, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_double, dptr, ctypes.c_int]
    return L


def _run(L, q, k, v, off, alpha, inv_n):
    total, heads, d = q.shape
    out = np.zeros((total, heads, d))
    P = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))
    L.hstu_oracle_fwd_f64(P(q, ctypes.c_float), P(k, ctypes.c_float), P(v, ctypes.c_float),
                          P(off, ctypes.c_int64), len(off) - 1, heads, d, alpha, inv_n,
                          P(out, ctypes.c_double), 2)
    return out


def _pins_pass(L) -> bool:
    """A condensed run of the pins: brute force, large-alpha limit, row-0 closed form."""
    rng = np.random.default_rng(0)
    lengths = [9, 0, 21, 1]
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T, H, d = int(off[-1]), 2, 8
    q, k, v = (rng.standard_normal((T, H, d)).astype(np.float32) for _ in range(3))
    ok = True
    got = _run(L, q, k, v, off, 0.4, 0.25)
    ref = dense.hstu_jagged_bruteforce(q, k, v, off, 0.4, 0.25)
    ok &= bool(np.allclose(got, ref, rtol=1e-12, atol=1e-13))
    qi, ki = (rng.integers(-3, 4, (T, H, d)).astype(np.float32) for _ in range(2))
    lim = _run(L, qi, ki, v, off, 200.0, 1.0) / 200.0
    for b in range(len(lengths)):
        s0, s1 = off[b], off[b + 1]
        for h in range(H):
            S = qi[s0:s1, h].astype(np.float64) @ ki[s0:s1, h].astype(np.float64).T
            ok &= bool(np.allclose(lim[s0:s1, h], np.tril(np.maximum(S, 0)) @ v[s0:s1, h], atol=1e-9))
    for b in range(len(lengths)):
        if lengths[b]:
            t = off[b]
            s = float(np.dot(q[t, 0].astype(np.float64), k[t, 0].astype(np.float64)))
            ok &= bool(np.allclose(got[t, 0], 0.25 * 0.4 * s * expit(0.4 * s) * v[t, 0], rtol=1e-12))
    return ok


def test_unmutated_copy_passes(tmp_path):
    src = open(oracle_build.SRC).read()
    (tmp_path / "orig.c").write_text(src)
    lib = tmp_path / "orig.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", str(lib),
                    str(tmp_path / "orig.c"), "-lm", "-lpthread"], check=True)
    L = ctypes.CDLL(str(lib))
    f, dptr, i64 = (ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                    ctypes.POINTER(ctypes.c_int64))
    L.hstu_oracle_fwd_f64.argtypes = [f, f, f, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_double, dptr, ctypes.c_int]
    assert _pins_pass(L)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert not _pins_pass(_build_mutant(tmp_path, name))


# ------------------------------------------------ the candidate (M-FALCON) mask
TARGET_MUTANTS = {
    "drop_self_term": ("return j <= i && (j < hist || j == i);", "return j <= i && (j < hist);"),
    "history_off_by_one": ("return j <= i && (j < hist || j == i);",
                           "return j <= i && (j <= hist || j == i);"),
    "candidates_see_each_other": ("return j <= i && (j < hist || j == i);", "return j <= i;"),
}


def _targets_pins_pass(L) -> bool:
    """Separate causal passes (the committed causal oracle) and the closed form
    of a candidates-only sequence, as in test_oracle_targets.py."""
    from oracle import reference
    f, dptr, i64 = (ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                    ctypes.POINTER(ctypes.c_int64))
    L.hstu_oracle_fwd_targets_f64.argtypes = [f, f, f, i64, i64, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_double, ctypes.c_double, dptr,
                                              ctypes.c_int]
    P = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))

    def run(q, k, v, off, nt, alpha, inv_n):
        total, heads, d = q.shape
        out = np.zeros((total, heads, d))
        off = np.asarray(off, dtype=np.int64)
        nt = np.asarray(nt, dtype=np.int64)
        L.hstu_oracle_fwd_targets_f64(P(q, ctypes.c_float), P(k, ctypes.c_float),
                                      P(v, ctypes.c_float), P(off, ctypes.c_int64),
                                      P(nt, ctypes.c_int64), len(off) - 1, heads, d, alpha, inv_n,
                                      P(out, ctypes.c_double), 2)
        return out

    rng = np.random.default_rng(5)
    hist, bm, H, d = 11, 5, 2, 8
    q, k, v = (rng.standard_normal((hist + bm, H, d)).astype(np.float32) for _ in range(3))
    got = run(q, k, v, [0, hist + bm], [bm], 0.6, 0.1)
    ok = True
    for c in range(bm):
        idx = list(range(hist)) + [hist + c]
        sub = reference.hstu_fwd(q[idx], k[idx], v[idx], [0, hist + 1], 0.6, 0.1)
        ok &= bool(np.allclose(got[hist + c], sub[hist], rtol=1e-12, atol=1e-14))
    only = run(q, k, v, [0, hist + bm], [hist + bm], 0.6, 0.1)
    s = 0.6 * np.einsum("thc,thc->th", q.astype(np.float64), k.astype(np.float64))
    ok &= bool(np.allclose(only, 0.1 * (s * expit(s))[..., None] * v, rtol=1e-12, atol=1e-14))
    return ok


def _build(tmp_path, name, src):
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    lib = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", str(lib), str(path),
                    "-lm", "-lpthread"], check=True)
    return ctypes.CDLL(str(lib))


def test_unmutated_copy_passes_the_candidate_pins(tmp_path):
    assert _targets_pins_pass(_build(tmp_path, "orig_t", open(oracle_build.SRC).read()))


@pytest.mark.parametrize("name", sorted(TARGET_MUTANTS))
def test_candidate_mutant_is_caught(tmp_path, name):
    src = open(oracle_build.SRC).read()
    old, new = TARGET_MUTANTS[name]
    assert src.count(old) == 1
    assert not _targets_pins_pass(_build(tmp_path, name, src.replace(old, new)))


# ------------------------------------------------ the output stage Norm(A V) (.) U
NORM_MUTANTS = {
    "unbiased_variance": ("var /= (double)width;", "var /= (double)(width - 1);"),
    "eps_outside_sqrt": ("1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)"),
    "mean_not_subtracted": ("(xr[c] - mean) * rstd", "xr[c] * rstd"),
    "beta_dropped": ("* (double)gamma[c] + (double)beta[c]", "* (double)gamma[c]"),
    "gate_by_first_column": ("(double)u[r * width + c]", "(double)u[r * width]"),
    "gamma_per_row": ("(double)gamma[c]", "(double)gamma[r % width]"),
}


def _norm_pins_pass(L) -> bool:
    """torch's layer_norm times u, as in test_oracle_norm_gate.py."""
    import torch
    f, dptr, i64 = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double), ctypes.c_int64
    L.hstu_oracle_norm_gate_f64.argtypes = [dptr, f, f, f, ctypes.c_double, i64, i64, dptr]
    P = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))
    rng = np.random.default_rng(12)
    rows, width, eps = 6, 16, 1e-2
    x = rng.standard_normal((rows, width)) * 0.3 + 0.5
    u = rng.standard_normal((rows, width)).astype(np.float32)
    g = (1.0 + 0.3 * rng.standard_normal(width)).astype(np.float32)
    b = (0.3 * rng.standard_normal(width)).astype(np.float32)
    y = np.zeros_like(x)
    L.hstu_oracle_norm_gate_f64(P(x, ctypes.c_double), P(u, ctypes.c_float), P(g, ctypes.c_float),
                                P(b, ctypes.c_float), eps, rows, width, P(y, ctypes.c_double))
    want = torch.nn.functional.layer_norm(torch.tensor(x), (width,), torch.tensor(g, dtype=torch.float64),
                                          torch.tensor(b, dtype=torch.float64), eps).numpy() * u
    return bool(np.abs(y - want).max() <= 1e-12 * np.abs(want).max())


def test_unmutated_copy_passes_the_norm_pins(tmp_path):
    assert _norm_pins_pass(_build(tmp_path, "orig_n", open(oracle_build.SRC).read()))


@pytest.mark.parametrize("name", sorted(NORM_MUTANTS))
def test_norm_mutant_is_caught(tmp_path, name):
    src = open(oracle_build.SRC).read()
    old, new = NORM_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    assert not _norm_pins_pass(_build(tmp_path, name, src.replace(old, new)))


# ------------------------------------------------ the relative attention bias rab_{p,t}
RAB_MUTANTS = {
    "bucket_of_delta_not_delta_plus_one": ("floor_log2_u64((uint64_t)delta + 1)",
                                           "floor_log2_u64((uint64_t)delta + (delta == 0))"),
    "time_difference_reversed": ("R->ts[seq_start + i] - R->ts[seq_start + j]",
                                 "R->ts[seq_start + j] - R->ts[seq_start + i]"),
    "candidates_keep_their_position": ("pi = i < hist ? i : hist", "pi = i"),
    "bias_scaled_by_alpha": ("hstu_oracle_silu(alpha * dot + bias)",
                             "hstu_oracle_silu(alpha * (dot + bias))"),
    "time_table_by_position_bucket": ("return (double)R->pos[bp] + (double)R->time[bt];",
                                      "return (double)R->pos[bp] + (double)R->time[bp < R->ntime ? bp : 0];"),
}


def _rab_pins_pass(L) -> bool:
    """Brute force with numpy-built buckets and the candidate identity, as in
    test_oracle_rab.py, through the planted copy."""
    from tests.test_oracle_rab import _bruteforce, _case, _tables
    f, dptr, i64 = (ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                    ctypes.POINTER(ctypes.c_int64))
    L.hstu_oracle_fwd_rab_f64.argtypes = [f, f, f, i64, i64, i64, f, ctypes.c_int, f, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                          ctypes.c_double, dptr, ctypes.c_int]
    P = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))

    def run(q, k, v, off, nt, ts, pos, time, alpha, inv_n):
        total, heads, d = q.shape
        out = np.zeros((total, heads, d))
        off = np.asarray(off, dtype=np.int64)
        keep = None if nt is None else np.asarray(nt, dtype=np.int64)
        ntp = None if keep is None else P(keep, ctypes.c_int64)
        ts = np.asarray(ts, dtype=np.int64)
        L.hstu_oracle_fwd_rab_f64(P(q, ctypes.c_float), P(k, ctypes.c_float), P(v, ctypes.c_float),
                                  P(off, ctypes.c_int64), ntp, P(ts, ctypes.c_int64),
                                  P(pos, ctypes.c_float), len(pos), P(time, ctypes.c_float),
                                  len(time), len(off) - 1, heads, d, alpha, inv_n,
                                  P(out, ctypes.c_double), 2)
        return out

    ok = True
    rng = np.random.default_rng(21)
    q, k, v, off, ts = _case(rng, [40, 25], 2, 8)
    pos, time = _tables(rng, 32, 32)
    nt = [11, 0]
    got = run(q, k, v, off, nt, ts, pos, time, 0.4, 0.05)
    want = _bruteforce(q, k, v, off, ts, pos, time, 0.4, 0.05, nt)
    ok &= bool(np.abs(got - want).max() <= 1e-12 * np.abs(want).max())
    return ok


def test_unmutated_copy_passes_the_rab_pins(tmp_path):
    assert _rab_pins_pass(_build(tmp_path, "orig_r", open(oracle_build.SRC).read()))


@pytest.mark.parametrize("name", sorted(RAB_MUTANTS))
def test_rab_mutant_is_caught(tmp_path, name):
    src = open(oracle_build.SRC).read()
    old, new = RAB_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    assert not _rab_pins_pass(_build(tmp_path, name, src.replace(old, new)))


# ------------------------------------------------ the backward pass
BWD_MUTANTS = {
    "silu_derivative_first_term_only": ("sg * (1.0 + x * (1.0 - sg)) * dp", "sg * dp"),
    "dv_without_inv_n": ("*p_out = J->inv_n * x * sg;", "*p_out = x * sg;"),
    "dk_from_k": ("dkj[c] += J->alpha * ds * (double)qi[c];", "dkj[c] += J->alpha * ds * (double)kj[c];"),
    "dq_without_alpha": ("dqi[c] += J->alpha * ds * (double)kj[c];", "dqi[c] += ds * (double)kj[c];"),
    "dp_from_q": ("dp += (double)doi[c] * (double)vj[c];", "dp += (double)doi[c] * (double)qi[c];"),
}


def _bwd_pins_pass(L) -> bool:
    """torch autograd of the dense definition, as in test_oracle_bwd.py."""
    from tests.test_oracle_bwd import _case, _dense_torch
    f, dptr, i64 = (ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                    ctypes.POINTER(ctypes.c_int64))
    L.hstu_oracle_bwd_f64.argtypes = [f, f, f, f, i64, i64, i64, f, ctypes.c_int, f, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                      ctypes.c_double, dptr, dptr, dptr, dptr, dptr, ctypes.c_int]
    P = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))
    rng = np.random.default_rng(31)
    q, k, v, do, off = _case(rng, [13, 20], 2, 8)
    off = off.astype(np.int64)
    grads = [np.zeros(q.shape) for _ in range(3)]
    L.hstu_oracle_bwd_f64(P(q, ctypes.c_float), P(k, ctypes.c_float), P(v, ctypes.c_float),
                          P(do, ctypes.c_float), P(off, ctypes.c_int64), None, None, None, 0, None, 0,
                          len(off) - 1, q.shape[1], q.shape[2], 0.4, 0.05,
                          *(P(g, ctypes.c_double) for g in grads), None, None, 2)
    want = _dense_torch(q, k, v, do, off, 0.4, 0.05)
    return all(np.abs(g - w_).max() <= 1e-12 * max(1.0, np.abs(w_).max()) for g, w_ in zip(grads, want))


def test_unmutated_copy_passes_the_bwd_pins(tmp_path):
    assert _bwd_pins_pass(_build(tmp_path, "orig_b", open(oracle_build.SRC).read()))


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_mutant_is_caught(tmp_path, name):
    src = open(oracle_build.SRC).read()
    old, new = BWD_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    assert not _bwd_pins_pass(_build(tmp_path, name, src.replace(old, new)))


# The bias tables' gradients: each mutant plants a plausible mistake in the
# per-pair sums; the pin is torch autograd of the dense definition with the
# tables as parameters (tests/test_oracle_bwd.py).  Both tables have 32
# entries here, so a bucket of one table always indexes the other in bounds.
TABLE_GRAD_MUTANTS = {
    "table_grads_from_p": ("gp[bp] += ds;", "gp[bp] += p;"),
    "time_grads_by_position_bucket": ("gt[bt] += ds;", "gt[bp] += ds;"),
    "table_grads_scaled_by_alpha": ("gp[bp] += ds;", "gp[bp] += J->alpha * ds;"),
}


def _table_grad_pins_pass(L) -> bool:
    from tests.test_oracle_bwd import dense_torch_rab, rab_case
    f, dptr, i64 = (ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                    ctypes.POINTER(ctypes.c_int64))
    L.hstu_oracle_bwd_f64.argtypes = [f, f, f, f, i64, i64, i64, f, ctypes.c_int, f, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                      ctypes.c_double, dptr, dptr, dptr, dptr, dptr, ctypes.c_int]
    P = lambda a, t: a.ctypes.data_as(ctypes.POINTER(t))
    rng = np.random.default_rng(33)
    q, k, v, do, off, ts, pos, time = rab_case(rng, [30, 17, 41], 2, 8, 32, 32)
    off = off.astype(np.int64)
    grads = [np.zeros(q.shape) for _ in range(3)] + [np.zeros(32), np.zeros(32)]
    rc = L.hstu_oracle_bwd_f64(P(q, ctypes.c_float), P(k, ctypes.c_float), P(v, ctypes.c_float),
                               P(do, ctypes.c_float), P(off, ctypes.c_int64), None,
                               P(ts, ctypes.c_int64), P(pos, ctypes.c_float), 32,
                               P(time, ctypes.c_float), 32, len(off) - 1, q.shape[1], q.shape[2],
                               0.4, 0.05, *(P(g, ctypes.c_double) for g in grads), 2)
    assert rc == 0
    want = dense_torch_rab(q, k, v, do, off, ts, pos, time, 0.4, 0.05)
    return all(np.abs(g - w_).max() <= 1e-12 * max(1.0, np.abs(w_).max()) for g, w_ in zip(grads, want))


def test_unmutated_copy_passes_the_table_grad_pins(tmp_path):
    assert _table_grad_pins_pass(_build(tmp_path, "orig_g", open(oracle_build.SRC).read()))


@pytest.mark.parametrize("name", sorted(TABLE_GRAD_MUTANTS))
def test_table_grad_mutant_is_caught(tmp_path, name):
    src = open(oracle_build.SRC).read()
    old, new = TABLE_GRAD_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    assert not _table_grad_pins_pass(_build(tmp_path, name, src.replace(old, new)))
