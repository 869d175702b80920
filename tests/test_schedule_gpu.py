"""GPU: the backward under its host-built per-CTA schedule.

The backward's CTAs run the items of a list schedule (each item, in
longest-first order, on the CTA free first) instead of every grid-th item.
On the skewed workload, where the schedule moves the most items, the
gradients are checked against the fp64 oracle on sampled rows, and a plan's
dK and dV equal a one-shot call's bit for bit (each comes from one CTA).
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
    yield
    parity.assert_device_ok()


def test_scheduled_backward_skewed_sampled_and_plan_equals_one_shot():
    w = workloads.workload("skewed")
    q, k, v = workloads.draw_qkv(w)
    rng = np.random.default_rng(4100)
    do = workloads.bf16_round((0.5 * rng.standard_normal(q.shape)).astype(np.float32))
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    a = [torch.empty_like(qd) for _ in range(3)]
    binding.hstu_attn_bwd(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                          w.inv_n, *a)
    g = [torch.empty_like(qd) for _ in range(3)]
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)
    try:
        binding.hstu_attn_bwd_plan(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    assert torch.equal(g[1], a[1]) and torch.equal(g[2], a[2])
    rt, rh, nu = parity.sample_rows(w, 128, seed=11)
    refs = reference.hstu_bwd_rows(q, k, v, do, w.offsets, w.alpha, w.inv_n, rt, rh)
    idx_t, idx_h = torch.as_tensor(rt, device="cuda"), torch.as_tensor(rh, device="cuda")
    for name, gt, rf in zip(("dq", "dk", "dv"), g, refs):
        got = gt[idx_t, idx_h].float().cpu().numpy().astype(np.float64)
        rms = float(np.sqrt(np.mean(rf[:nu] ** 2)))
        worst = float(parity.ratio(got, rf, rms).max())
        assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f}"
