"""GPU parity of the backward pass against the fp64 oracle.

HSTU paper Appendix G: the backward recomputes the attention; the
gradients dq, dk, dv of sum(out * dout) are those of the forward definition
(oracle.reference.hstu_bwd).  Every element of each gradient must satisfy
the bound of tests/parity.py, with that gradient's own rms.
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


LENGTHS = [300, 513, 256, 700, 90, 129, 0, 1, 640, 385]


def _run(w, seed, dscale=1.0):
    q, k, v = workloads.draw_qkv(w, seed=seed)
    rng = np.random.default_rng(seed + 1)
    do = workloads.bf16_round((dscale * rng.standard_normal(q.shape)).astype(np.float32))
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
    binding.hstu_attn_bwd(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                          w.inv_n, dq, dk, dv)
    torch.cuda.synchronize()
    parity.assert_device_ok()
    ref = reference.hstu_bwd(q, k, v, do, w.offsets, w.alpha, w.inv_n)
    return (dq, dk, dv), ref


def _check(got, ref, name):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    r = parity.ratio(g, ref, rms)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f} at {np.unravel_index(r.argmax(), r.shape)}"


@pytest.mark.parametrize("d", [32, 64, 128])
def test_bwd_full_parity(d):
    w = workloads.custom(LENGTHS, heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    got, ref = _run(w, seed=800 + d)
    for gt, rf, name in zip(got, ref, ("dq", "dk", "dv")):
        _check(gt, rf, name)


def test_bwd_long_sequences():
    w = workloads.custom([2048, 1500], heads=2, d=64)
    got, ref = _run(w, seed=850)
    for gt, rf, name in zip(got, ref, ("dq", "dk", "dv")):
        _check(gt, rf, name)


def test_bwd_is_deterministic_in_dk_dv_and_close_in_dq():
    # dk and dv come from one CTA each: bit-identical on a rerun; dq sums
    # parts with atomics, whose order may differ
    w = workloads.custom([700, 129], heads=2, d=64)
    (a, _) = _run(w, seed=860)
    (b, _) = _run(w, seed=860)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2 * a[0].float().abs().max().item()


def test_bwd_plan_equals_one_shot():
    w = workloads.custom(LENGTHS, heads=2, d=64)
    (a, _) = _run(w, seed=870)
    q, k, v = workloads.draw_qkv(w, seed=870)
    rng = np.random.default_rng(871)
    do = workloads.bf16_round(rng.standard_normal(q.shape).astype(np.float32))
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    g = [torch.empty_like(qd) for _ in range(3)]
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)
    try:
        binding.hstu_attn_bwd_plan(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g)
        binding.hstu_attn_bwd_plan(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g)  # the accumulator restarts
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    assert torch.equal(g[1], a[1]) and torch.equal(g[2], a[2])
    assert (g[0].float() - a[0].float()).abs().max().item() <= 1e-2 * a[0].float().abs().max().item()
    parity.assert_device_ok()


def test_bwd_dense_workload_sampled():
    # full size, in the launch configuration the benchmark times (a plan)
    w = workloads.workload("dense")
    q, k, v = workloads.draw_qkv(w)
    rng = np.random.default_rng(4000 + w.index)
    do = workloads.bf16_round(rng.standard_normal(q.shape).astype(np.float32))
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    g = [torch.empty_like(qd) for _ in range(3)]
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)
    try:
        binding.hstu_attn_bwd_plan(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    rt, rh, nu = parity.sample_rows(w, 192, seed=7)
    refs = reference.hstu_bwd_rows(q, k, v, do, w.offsets, w.alpha, w.inv_n, rt, rh)
    idx_t, idx_h = torch.as_tensor(rt, device="cuda"), torch.as_tensor(rh, device="cuda")
    for name, gt, rf in zip(("dq", "dk", "dv"), g, refs):
        got = gt[idx_t, idx_h].float().cpu().numpy().astype(np.float64)
        rms = float(np.sqrt(np.mean(rf[:nu] ** 2)))
        assert np.all(np.isfinite(got)), name
        worst = parity.ratio(got, rf, rms).max()
        assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f}"
