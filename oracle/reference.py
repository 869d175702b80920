"""ctypes wrapper of the fp64 C oracle (``hstu_oracle.c``).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The oracle evaluates, for each sequence b, head h and local row i
(ai6s.net "HSTU fused operator" post, section 1 formula; section 3.2 tril
block mask including the diagonal; section 4.2 jagged values + offsets):

    out[t, h, :] = inv_n * sum_{j <= i} silu(alpha * q[t,h,:].k[off[b]+j,h,:]) * v[off[b]+j,h,:]

With ``num_targets`` (HSTU paper section 3.4 and Appendix H, Algorithm 1:
the M-FALCON mask), the last num_targets[b] tokens of sequence b are
candidates: term j of row i is kept iff j <= i and (j < hist or j == i),
hist = n_b - num_targets[b].

With ``rab`` = (ts, pos, time) -- one timestamp per token and two bias
tables -- the scores get the relative attention bias of the HSTU paper
(section 3, rab_{p,t}; reading in hstu_oracle.c): silu(alpha q.k + pos[bp]
+ time[bt]), bp and bt the clipped floor(log2(delta + 1)) buckets of the
relative position (candidates sit at position hist) and of the timestamp
difference (clamped at 0).

``norm_gate`` is the layer's output stage on those rows, Norm(A V) (.) U
(HSTU paper section 3 and section 3.1): a layer norm over each token's
heads * d outputs with affine gamma, beta, times U elementwise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        f = ctypes.POINTER(ctypes.c_float)
        d = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.POINTER(ctypes.c_int64)
        i32 = ctypes.POINTER(ctypes.c_int32)
        lib.hstu_oracle_silu.argtypes = [ctypes.c_double]
        lib.hstu_oracle_silu.restype = ctypes.c_double
        lib.hstu_oracle_fwd_f64.argtypes = [f, f, f, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_double, d, ctypes.c_int]
        lib.hstu_oracle_fwd_f64.restype = ctypes.c_int
        lib.hstu_oracle_rows_f64.argtypes = [f, f, f, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_double, ctypes.c_double, i64, i32,
                                             ctypes.c_int64, d, ctypes.c_int]
        lib.hstu_oracle_rows_f64.restype = ctypes.c_int
        lib.hstu_oracle_fwd_targets_f64.argtypes = [f, f, f, i64, i64, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                                    d, ctypes.c_int]
        lib.hstu_oracle_fwd_targets_f64.restype = ctypes.c_int
        lib.hstu_oracle_rows_targets_f64.argtypes = [f, f, f, i64, i64, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                                     i64, i32, ctypes.c_int64, d, ctypes.c_int]
        lib.hstu_oracle_rows_targets_f64.restype = ctypes.c_int
        lib.hstu_oracle_norm_gate_f64.argtypes = [d, f, f, f, ctypes.c_double, ctypes.c_int64,
                                                  ctypes.c_int64, d]
        lib.hstu_oracle_norm_gate_f64.restype = ctypes.c_int
        lib.hstu_oracle_rab_bucket.argtypes = [ctypes.c_int64, ctypes.c_int]
        lib.hstu_oracle_rab_bucket.restype = ctypes.c_int
        lib.hstu_oracle_fwd_rab_f64.argtypes = [f, f, f, i64, i64, i64, f, ctypes.c_int, f,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_double, ctypes.c_double, d,
                                                ctypes.c_int]
        lib.hstu_oracle_fwd_rab_f64.restype = ctypes.c_int
        lib.hstu_oracle_rows_rab_f64.argtypes = [f, f, f, i64, i64, i64, f, ctypes.c_int, f,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_double, ctypes.c_double, i64,
                                                 i32, ctypes.c_int64, d, ctypes.c_int]
        lib.hstu_oracle_rows_rab_f64.restype = ctypes.c_int
        lib.hstu_oracle_bwd_f64.argtypes = [f, f, f, f, i64, i64, i64, f, ctypes.c_int, f,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_double, d, d, d, d, d,
                                            ctypes.c_int]
        lib.hstu_oracle_bwd_f64.restype = ctypes.c_int
        lib.hstu_oracle_bwd_rows_f64.argtypes = [f, f, f, f, i64, i64, i64, f, ctypes.c_int, f,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_double, ctypes.c_double, i64,
                                                 i32, ctypes.c_int64, d, d, d]
        lib.hstu_oracle_bwd_rows_f64.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _f32(x) -> np.ndarray:
    """Accept a torch tensor (any float dtype, incl. bf16) or numpy array -> contiguous fp32."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def silu(x: float) -> float:
    """The oracle's own silu, exposed for pinning."""
    return _load().hstu_oracle_silu(float(x))


def rab_bucket(delta: int, nbuckets: int) -> int:
    """The oracle's bias bucket min(floor(log2(max(delta, 0) + 1)), nbuckets - 1), for pinning."""
    return _load().hstu_oracle_rab_bucket(int(delta), int(nbuckets))


def _rab_arrays(rab, total):
    ts, pos, time = rab
    ts = np.ascontiguousarray(np.asarray(ts), dtype=np.int64).reshape(-1)
    pos, time = _f32(pos).reshape(-1), _f32(time).reshape(-1)
    if ts.shape != (total,) or pos.size < 1 or time.size < 1:
        raise ValueError("rab needs one timestamp per token and non-empty tables")
    return ts, pos, time


def _targets_ptr(num_targets, batch):
    if num_targets is None:
        return None, None
    nt = np.ascontiguousarray(np.asarray(num_targets), dtype=np.int64)
    if nt.shape != (batch,):
        raise ValueError("num_targets needs one entry per sequence")
    return nt, _ptr(nt, ctypes.c_int64)


def hstu_fwd(q, k, v, offsets, alpha: float, inv_n: float, threads: int | None = None,
             num_targets=None, rab=None) -> np.ndarray:
    """All rows: returns fp64 array (total, heads, d)."""
    qf, kf, vf = _f32(q), _f32(k), _f32(v)
    total, heads, d = qf.shape
    off = np.ascontiguousarray(np.asarray(offsets), dtype=np.int64)
    batch = len(off) - 1
    if kf.shape != qf.shape or vf.shape != qf.shape or (batch >= 0 and off[-1] != total):
        raise ValueError("shape mismatch between q/k/v/offsets")
    out = np.zeros((total, heads, d), dtype=np.float64)
    if rab is not None:
        ts, pos, time = _rab_arrays(rab, total)
        nt, ntp = _targets_ptr(num_targets, batch)
        rc = _load().hstu_oracle_fwd_rab_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                             _ptr(vf, ctypes.c_float), _ptr(off, ctypes.c_int64), ntp,
                                             _ptr(ts, ctypes.c_int64), _ptr(pos, ctypes.c_float),
                                             pos.size, _ptr(time, ctypes.c_float), time.size, batch,
                                             heads, d, float(alpha), float(inv_n),
                                             _ptr(out, ctypes.c_double), threads or default_threads())
    elif num_targets is None:
        rc = _load().hstu_oracle_fwd_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                         _ptr(vf, ctypes.c_float), _ptr(off, ctypes.c_int64),
                                         batch, heads, d, float(alpha), float(inv_n),
                                         _ptr(out, ctypes.c_double), threads or default_threads())
    else:
        nt = np.ascontiguousarray(np.asarray(num_targets), dtype=np.int64)
        if nt.shape != (batch,):
            raise ValueError("num_targets needs one entry per sequence")
        rc = _load().hstu_oracle_fwd_targets_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                                 _ptr(vf, ctypes.c_float), _ptr(off, ctypes.c_int64),
                                                 _ptr(nt, ctypes.c_int64), batch, heads, d,
                                                 float(alpha), float(inv_n),
                                                 _ptr(out, ctypes.c_double),
                                                 threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments (offsets must start at 0 and not decrease; "
                         "0 <= num_targets <= length)")
    return out


def hstu_rows(q, k, v, offsets, alpha: float, inv_n: float, rows_t, rows_h,
              threads: int | None = None, num_targets=None, rab=None) -> np.ndarray:
    """Sampled rows: row r is (token rows_t[r], head rows_h[r]); returns fp64 (nrows, d)."""
    qf, kf, vf = _f32(q), _f32(k), _f32(v)
    total, heads, d = qf.shape
    off = np.ascontiguousarray(np.asarray(offsets), dtype=np.int64)
    rt = np.ascontiguousarray(rows_t, dtype=np.int64)
    rh = np.ascontiguousarray(rows_h, dtype=np.int32)
    if rt.shape != rh.shape:
        raise ValueError("rows_t and rows_h differ in length")
    out = np.zeros((len(rt), d), dtype=np.float64)
    if rab is not None:
        ts, pos, time = _rab_arrays(rab, total)
        nt, ntp = _targets_ptr(num_targets, len(off) - 1)
        rc = _load().hstu_oracle_rows_rab_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                              _ptr(vf, ctypes.c_float), _ptr(off, ctypes.c_int64),
                                              ntp, _ptr(ts, ctypes.c_int64),
                                              _ptr(pos, ctypes.c_float), pos.size,
                                              _ptr(time, ctypes.c_float), time.size, len(off) - 1,
                                              heads, d, float(alpha), float(inv_n),
                                              _ptr(rt, ctypes.c_int64), _ptr(rh, ctypes.c_int32),
                                              len(rt), _ptr(out, ctypes.c_double),
                                              threads or default_threads())
    elif num_targets is None:
        rc = _load().hstu_oracle_rows_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                          _ptr(vf, ctypes.c_float), _ptr(off, ctypes.c_int64),
                                          len(off) - 1, heads, d, float(alpha), float(inv_n),
                                          _ptr(rt, ctypes.c_int64), _ptr(rh, ctypes.c_int32), len(rt),
                                          _ptr(out, ctypes.c_double), threads or default_threads())
    else:
        nt = np.ascontiguousarray(np.asarray(num_targets), dtype=np.int64)
        if nt.shape != (len(off) - 1,):
            raise ValueError("num_targets needs one entry per sequence")
        rc = _load().hstu_oracle_rows_targets_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                                  _ptr(vf, ctypes.c_float), _ptr(off, ctypes.c_int64),
                                                  _ptr(nt, ctypes.c_int64), len(off) - 1, heads, d,
                                                  float(alpha), float(inv_n), _ptr(rt, ctypes.c_int64),
                                                  _ptr(rh, ctypes.c_int32), len(rt),
                                                  _ptr(out, ctypes.c_double), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def norm_gate(x, u, gamma, beta, eps: float) -> np.ndarray:
    """Layer norm over the last two axes of x (heads * d per token), affine
    gamma/beta of that width, times u elementwise.  x: (rows, heads, d) any
    float type (taken as fp64); u: same shape; returns fp64."""
    xf = np.ascontiguousarray(x, dtype=np.float64)
    if xf.ndim != 3:
        raise ValueError("x must be (rows, heads, d)")
    rows, heads, d = xf.shape
    uf = _f32(u)
    g, b = _f32(gamma).reshape(-1), _f32(beta).reshape(-1)
    if uf.shape != xf.shape or g.shape != (heads * d,) or b.shape != (heads * d,):
        raise ValueError("u must match x and gamma/beta must have heads * d entries")
    y = np.zeros_like(xf)
    rc = _load().hstu_oracle_norm_gate_f64(_ptr(xf, ctypes.c_double), _ptr(uf, ctypes.c_float),
                                           _ptr(g, ctypes.c_float), _ptr(b, ctypes.c_float),
                                           float(eps), rows, heads * d, _ptr(y, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (eps must be >= 0)")
    return y


def hstu_fwd_norm_gate(q, k, v, u, gamma, beta, eps: float, offsets, alpha: float, inv_n: float,
                       threads: int | None = None, num_targets=None, rab=None) -> np.ndarray:
    """Norm(A V) (.) U over all tokens: fp64 (total, heads, d)."""
    x = hstu_fwd(q, k, v, offsets, alpha, inv_n, threads=threads, num_targets=num_targets, rab=rab)
    return norm_gate(x, u, gamma, beta, eps)


def hstu_rows_norm_gate(q, k, v, u, gamma, beta, eps: float, offsets, alpha: float, inv_n: float,
                        rows_t, threads: int | None = None, num_targets=None, rab=None) -> np.ndarray:
    """Norm(A V) (.) U for the sampled tokens rows_t: fp64 (nrows, heads, d)."""
    heads, d = np.shape(q)[1], np.shape(q)[2]
    rt = np.repeat(np.asarray(rows_t, dtype=np.int64), heads)
    rh = np.tile(np.arange(heads, dtype=np.int32), len(rows_t))
    x = hstu_rows(q, k, v, offsets, alpha, inv_n, rt, rh, threads=threads,
                  num_targets=num_targets, rab=rab).reshape(len(rows_t), heads, d)
    return norm_gate(x, _f32(u)[np.asarray(rows_t, dtype=np.int64)], gamma, beta, eps)


def hstu_bwd(q, k, v, dout, offsets, alpha: float, inv_n: float, threads: int | None = None,
             num_targets=None, rab=None, table_grads: bool = False):
    """Gradients of sum(out * dout) with respect to q, k, v: fp64 arrays
    (total, heads, d) each (HSTU paper Appendix G: the backward of the
    forward definition; the chain rule is written out in hstu_oracle.c).
    With ``rab`` and ``table_grads``, also the bias tables' gradients:
    returns (dq, dk, dv, dpos, dtime)."""
    qf, kf, vf, df = _f32(q), _f32(k), _f32(v), _f32(dout)
    total, heads, d = qf.shape
    off = np.ascontiguousarray(np.asarray(offsets), dtype=np.int64)
    batch = len(off) - 1
    if (kf.shape != qf.shape or vf.shape != qf.shape or df.shape != qf.shape
            or (batch >= 0 and off[-1] != total)):
        raise ValueError("shape mismatch between q/k/v/dout/offsets")
    nt, ntp = _targets_ptr(num_targets, batch)
    tsp = posp = timep = None
    npos = ntime = 0
    if rab is not None:
        ts, pos, time = _rab_arrays(rab, total)
        tsp, posp, timep = _ptr(ts, ctypes.c_int64), _ptr(pos, ctypes.c_float), _ptr(time, ctypes.c_float)
        npos, ntime = pos.size, time.size
    dq, dk, dv = (np.zeros((total, heads, d), dtype=np.float64) for _ in range(3))
    gpos = np.zeros(max(npos, 1)), np.zeros(max(ntime, 1))
    rc = _load().hstu_oracle_bwd_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                     _ptr(vf, ctypes.c_float), _ptr(df, ctypes.c_float),
                                     _ptr(off, ctypes.c_int64), ntp, tsp, posp, npos, timep, ntime,
                                     batch, heads, d, float(alpha), float(inv_n),
                                     _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                     _ptr(dv, ctypes.c_double), _ptr(gpos[0], ctypes.c_double),
                                     _ptr(gpos[1], ctypes.c_double), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    if rab is not None and table_grads:
        return dq, dk, dv, gpos[0][:npos], gpos[1][:ntime]
    return dq, dk, dv


def hstu_bwd_rows(q, k, v, dout, offsets, alpha: float, inv_n: float, rows_t, rows_h, rab=None,
                  num_targets=None):
    """Sampled gradient rows (``num_targets`` and ``rab`` as hstu_bwd): for row
    r = (token rows_t[r], head rows_h[r]) the fp64 dq, dk, dv rows, each
    (nrows, d)."""
    qf, kf, vf, df = _f32(q), _f32(k), _f32(v), _f32(dout)
    total, heads, d = qf.shape
    off = np.ascontiguousarray(np.asarray(offsets), dtype=np.int64)
    nt, ntp = _targets_ptr(num_targets, len(off) - 1)
    tsp = posp = timep = None
    npos = ntime = 0
    if rab is not None:
        ts, pos, time = _rab_arrays(rab, total)
        tsp, posp, timep = _ptr(ts, ctypes.c_int64), _ptr(pos, ctypes.c_float), _ptr(time, ctypes.c_float)
        npos, ntime = pos.size, time.size
    rt = np.ascontiguousarray(rows_t, dtype=np.int64)
    rh = np.ascontiguousarray(rows_h, dtype=np.int32)
    if rt.shape != rh.shape:
        raise ValueError("rows_t and rows_h differ in length")
    dq, dk, dv = (np.zeros((len(rt), d), dtype=np.float64) for _ in range(3))
    rc = _load().hstu_oracle_bwd_rows_f64(_ptr(qf, ctypes.c_float), _ptr(kf, ctypes.c_float),
                                          _ptr(vf, ctypes.c_float), _ptr(df, ctypes.c_float),
                                          _ptr(off, ctypes.c_int64), ntp, tsp, posp, npos, timep,
                                          ntime, len(off) - 1, heads, d,
                                          float(alpha), float(inv_n), _ptr(rt, ctypes.c_int64),
                                          _ptr(rh, ctypes.c_int32), len(rt), _ptr(dq, ctypes.c_double),
                                          _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return dq, dk, dv
