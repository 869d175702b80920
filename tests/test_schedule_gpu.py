"""GPU: the forward under the host-built per-CTA schedule.

Plans and one-shot calls run each CTA's items from a schedule built on the
host (list scheduling, in batches of (sequence, head) groups where the
operands exceed 48 MiB).  The no-allocation entry still takes the
longest-first list serpentine.  An item's rows are computed by one CTA from
the same operands whichever CTA runs it, so the two must agree bit for bit;
the scheduled result is also checked against the fp64 oracle on sampled
rows, and a plan's launch reports its schedule's grid.
"""
import numpy as np
import pytest
import torch

from hstu_jagged_attention_gb300 import binding, build, workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    yield
    parity.assert_device_ok()


def _batched_workload():
    # 24 x 8192 tokens, 4 heads, d = 64: 192 MiB of K and V, so the schedule
    # takes the groups in batches
    lengths = np.full(24, 8192)
    lengths[::5] = 5000
    lengths[3] = 1
    return workloads.custom(lengths, heads=4, d=64)


def test_scheduled_forward_equals_serpentine_bit_for_bit():
    w = _batched_workload()
    assert w.total * w.heads * w.d * 4 > 48 * (1 << 20)
    (q, k, v) = workloads.draw_qkv(w, seed=400)
    qd, kd, vd = parity.to_device(q, k, v)
    a = torch.empty_like(qd)
    binding.hstu_attn_fwd(qd, kd, vd, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha, w.inv_n, a)
    b = torch.empty_like(qd)
    binding.hstu_attn_fwd_noalloc(qd, kd, vd, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                  w.inv_n, b)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    parity.sampled_check(w, q, k, v, a, n_random=64, seed=4)
    assert binding.hstu_last_status() == (binding.HSTU_OK, 0)


def test_plan_launch_shape_is_the_schedule_grid():
    w = _batched_workload()
    plan = binding.hstu_plan_create(w.offsets, w.batch, w.heads, w.d, w.max_seqlen)
    try:
        grid, block, smem = binding.hstu_launch_shape(plan)
        n = binding.hstu_plan_num_items(plan)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert grid == min(n, sms) and block == 512 and smem > 0
    finally:
        binding.hstu_plan_destroy(plan)


def test_scheduled_candidates_plan_equals_one_shot():
    w, nt = workloads.candidate_workload()
    q, k, v = parity.to_device(*workloads.draw_qkv(w, seed=401))
    a = torch.empty_like(q)
    binding.hstu_attn_fwd_targets(q, k, v, w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                  w.inv_n, a)
    plan = binding.hstu_plan_create_targets(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen)
    try:
        b = torch.empty_like(q)
        binding.hstu_attn_fwd_plan(plan, q, k, v, w.alpha, w.inv_n, b)
    finally:
        binding.hstu_plan_destroy(plan)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.isfinite(a.float()).all()
