"""GPU parity of the backward with candidates (the M-FALCON mask).

HSTU paper section 3.4 and Appendix H: candidates see the history and
themselves only; Appendix G: the backward recomputes the attention.  The
gradients of sum(out * dout) under that mask (and with the bias) are
checked element by element against oracle.reference.hstu_bwd(...,
num_targets=...) with the bound of tests/parity.py, each with its own rms.
"""
import numpy as np
import pytest
import torch

from hstu_jagged_attention_gb300 import binding, build, workloads
from oracle import reference
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.hstu_set_wait_timeout_ns(0)
    yield
    parity.assert_device_ok()


# (length, candidates): history a multiple of 128, one candidate, all
# candidates, none, candidates spanning several key blocks
CASES = [(300, 100), (513, 128), (256, 1), (700, 333), (90, 90), (129, 0), (0, 0), (1, 1),
         (640, 500), (385, 2), (384, 128), (1000, 999)]
NAMES = ("dq", "dk", "dv", "dpos", "dtime")


def _inputs(w, seed):
    q, k, v = workloads.draw_qkv(w, seed=seed)
    rng = np.random.default_rng(seed + 1)
    do = workloads.bf16_round(rng.standard_normal(q.shape).astype(np.float32))
    return q, k, v, do


def _check(got, ref, name):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    r = parity.ratio(g, ref, rms)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f} at {np.unravel_index(r.argmax(), r.shape)}"


def _run(w, nt, q, k, v, do, rab=None):
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    g = [torch.empty_like(qd) for _ in range(3)]
    kw = {}
    if rab is not None:
        kw = dict(rab=tuple(torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in rab),
                  dpos=torch.empty(rab[1].size, device="cuda"),
                  dtime=torch.empty(rab[2].size, device="cuda"))
    binding.hstu_attn_bwd_ex(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                             w.inv_n, *g, num_targets=nt, **kw)
    torch.cuda.synchronize()
    parity.assert_device_ok()
    return g + ([kw["dpos"], kw["dtime"]] if rab is not None else [])


@pytest.mark.parametrize("d", [32, 64, 128])
def test_bwd_candidates_parity(d):
    w = workloads.custom([n for n, _ in CASES], heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    q, k, v, do = _inputs(w, 1600 + d)
    got = _run(w, nt, q, k, v, do)
    ref = reference.hstu_bwd(q, k, v, do, w.offsets, w.alpha, w.inv_n, num_targets=nt)
    for gt, rf, name in zip(got, ref, NAMES):
        _check(gt, rf, name)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_candidates_with_the_bias(d):
    w = workloads.custom([n for n, _ in CASES], heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    q, k, v, do = _inputs(w, 1650 + d)
    ts, pos, time = workloads.draw_rab(w, seed=1660 + d, backwards=0.1)
    rab = (ts, pos[:20].copy(), time[:27].copy())
    got = _run(w, nt, q, k, v, do, rab)
    ref = reference.hstu_bwd(q, k, v, do, w.offsets, w.alpha, w.inv_n, num_targets=nt, rab=rab,
                             table_grads=True)
    for gt, rf, name in zip(got, ref, NAMES):
        _check(gt, rf, name)


def test_bwd_zero_candidates_equal_the_causal_backward():
    # no candidate anywhere: the causal work list and masks, so dk and dv
    # equal the plain call's bit for bit
    w = workloads.custom([700, 1, 129, 256, 513], heads=2, d=64)
    q, k, v, do = _inputs(w, 1670)
    got = _run(w, np.zeros(w.batch, np.int32), q, k, v, do)
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    plain = [torch.empty_like(qd) for _ in range(3)]
    binding.hstu_attn_bwd(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                          w.inv_n, *plain)
    torch.cuda.synchronize()
    assert torch.equal(got[1], plain[1]) and torch.equal(got[2], plain[2])


def test_bwd_candidates_plan_equals_one_shot():
    w = workloads.custom([n for n, _ in CASES], heads=2, d=64)
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    q, k, v, do = _inputs(w, 1680)
    a = _run(w, nt, q, k, v, do)
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    g = [torch.empty_like(qd) for _ in range(3)]
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)
    try:
        binding.hstu_attn_bwd_plan(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    assert torch.equal(g[1], a[1]) and torch.equal(g[2], a[2])
    assert (g[0].float() - a[0].float()).abs().max().item() <= 1e-2 * a[0].float().abs().max().item()


def test_bwd_candidate_workload_sampled():
    # full size, in the launch configuration the benchmark times (a plan):
    # 32 histories of 2048..8192 tokens with 1024 candidates each
    w, nt = workloads.candidate_workload()
    q, k, v = workloads.draw_qkv(w)
    rng = np.random.default_rng(4000 + w.index)
    do = workloads.bf16_round(rng.standard_normal(q.shape).astype(np.float32))
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    g = [torch.empty_like(qd) for _ in range(3)]
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)
    try:
        binding.hstu_attn_bwd_plan(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    rt, rh, nu = parity.sample_rows(w, 192, seed=9)
    # and each of the first 8 sequences' last history row, first and last candidate
    off = w.offsets.astype(np.int64)
    extra = [t for b in range(8) for t in (off[b + 1] - nt[b] - 1, off[b + 1] - nt[b], off[b + 1] - 1)]
    rt = np.concatenate([rt, np.array(extra, dtype=rt.dtype)])
    rh = np.concatenate([rh, np.arange(len(extra), dtype=rh.dtype) % w.heads])
    refs = reference.hstu_bwd_rows(q, k, v, do, w.offsets, w.alpha, w.inv_n, rt, rh, num_targets=nt)
    idx_t, idx_h = torch.as_tensor(rt, device="cuda"), torch.as_tensor(rh, device="cuda")
    for name, gt, rf in zip(("dq", "dk", "dv"), g, refs):
        got = gt[idx_t, idx_h].float().cpu().numpy().astype(np.float64)
        rms = float(np.sqrt(np.mean(rf[:nu] ** 2)))
        assert np.all(np.isfinite(got)), name
        worst = parity.ratio(got, rf, rms).max()
        assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f}"
