"""Shared helpers for the GPU parity tests (not a test module).

Tolerance: every output element must satisfy
    |gpu - ref| <= 1e-2 * |ref| + 1e-3 * rms(ref)
where ref is the fp64 oracle on the same bf16 inputs and rms(ref) is the
root mean square of the reference output (over all elements when the whole
output is checked; over a uniform random sample of rows otherwise).
"""
from __future__ import annotations

import numpy as np
import torch

from hstu_jagged_attention_gb300 import binding, workloads
from oracle import reference

RTOL = 1e-2
RMS_TOL = 1e-3


def ratio(got: np.ndarray, ref: np.ndarray, rms: float) -> np.ndarray:
    """err / allowed, elementwise; parity holds where this is <= 1."""
    allowed = RTOL * np.abs(ref) + RMS_TOL * rms
    return np.abs(got - ref) / np.maximum(allowed, 1e-300)


def to_device(q, k, v):
    return tuple(t.to("cuda").contiguous() for t in (q, k, v))


def run_plan(w: workloads.Workload, q, k, v, out=None) -> torch.Tensor:
    """The launch configuration the benchmark times: a prebuilt plan, device buffers."""
    out = torch.empty_like(q) if out is None else out
    plan = binding.hstu_plan_create(w.offsets, w.batch, w.heads, w.d, w.max_seqlen)
    try:
        binding.hstu_attn_fwd_plan(plan, q, k, v, w.alpha, w.inv_n, out)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    return out


def run_call(w: workloads.Workload, q, k, v, offsets=None) -> torch.Tensor:
    out = torch.empty_like(q)
    binding.hstu_attn_fwd(q, k, v, w.offsets if offsets is None else offsets, w.batch, w.heads, w.d,
                          w.max_seqlen, w.alpha, w.inv_n, out)
    torch.cuda.synchronize()
    return out


def assert_device_ok():
    st, site = binding.hstu_last_status()
    assert st == binding.HSTU_OK, f"device wait gave up (site {site})"


def full_check(w, q, k, v, out) -> float:
    ref = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n)
    got = out.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    r = ratio(got, ref, rms)
    worst = float(r.max()) if r.size else 0.0
    assert np.all(np.isfinite(got)), "non-finite output"
    assert worst <= 1.0, f"parity fails: worst err/tol {worst:.3f} at {np.unravel_index(r.argmax(), r.shape)}"
    return worst


def sample_rows(w: workloads.Workload, n_random: int, seed: int = 0):
    """A uniform random sample of (token, head) rows plus edge rows.

    Returns (rows_t, rows_h, n_uniform): the first n_uniform rows are the
    uniform sample (used for the rms estimate), the rest are edge rows:
    first/last token of sequences, 128-row block boundaries, the longest
    sequence's last rows.
    """
    rng = np.random.default_rng(seed)
    T, H = w.total, w.heads
    ut = rng.integers(0, T, size=n_random)
    uh = rng.integers(0, H, size=n_random)
    off = w.offsets.astype(np.int64)
    edge_t = []
    order = np.argsort(-w.lengths)
    for b in list(order[:4]) + list(rng.choice(w.batch, size=min(6, w.batch), replace=False)):
        s0, n = int(off[b]), int(w.lengths[b])
        if n == 0:
            continue
        for i in {0, n - 1, min(127, n - 1), min(128, n - 1), (n - 1) // 128 * 128, max(n - 2, 0)}:
            edge_t.append(s0 + i)
    edge_t = np.array(sorted(set(edge_t)), dtype=np.int64)
    edge_h = rng.integers(0, H, size=len(edge_t))
    return np.concatenate([ut, edge_t]), np.concatenate([uh, edge_h]), n_random


def sampled_check(w, q, k, v, out, n_random=256, seed=0) -> float:
    rt, rh, nu = sample_rows(w, n_random, seed)
    ref = reference.hstu_rows(q, k, v, w.offsets, w.alpha, w.inv_n, rt, rh)
    got_all = out  # (T, H, d) on device
    idx_t = torch.as_tensor(rt, device=got_all.device)
    idx_h = torch.as_tensor(rh, device=got_all.device)
    got = got_all[idx_t, idx_h].float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref[:nu] ** 2)))
    r = ratio(got, ref, rms)
    worst = float(r.max())
    assert np.all(np.isfinite(got)), "non-finite output"
    assert worst <= 1.0, f"parity fails: worst err/tol {worst:.3f} at sampled row {r.max(axis=1).argmax()}"
    return worst
