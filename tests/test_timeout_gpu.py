"""Bounded device-side waits: a wait that runs out returns instead of hanging.

The kernel's waits are limited by %globaltimer.  The test hook
HSTU_DEBUG_UNSIGNALLED_WAIT makes the MMA warp wait on a barrier that
nothing signals; with a 1 ms limit that wait gives up, and the kernel must
then drain its own copies and MMAs, free TMEM and return, report
HSTU_ERR_TIMEOUT through hstu_last_status, and leave the context usable for
the next (normal) launch.  Nothing here faults or traps the GPU.
"""
import pytest
import torch

from hstu_jagged_attention_gb300 import binding, build, workloads
from tests import parity

pytestmark = pytest.mark.gpu


def test_wait_limit_gives_timeout_status_and_context_survives():
    build.build()
    w = workloads.custom([700, 300, 5], heads=2, d=64)
    q, k, v = parity.to_device(*workloads.draw_qkv(w, seed=21))
    binding.hstu_last_status()  # clear
    try:
        binding.hstu_set_wait_timeout_ns(1_000_000)
        binding.hstu_set_debug_flags(binding.HSTU_DEBUG_UNSIGNALLED_WAIT)
        out = torch.zeros_like(q)
        plan = binding.hstu_plan_create(w.offsets, w.batch, w.heads, w.d, w.max_seqlen)
        binding.hstu_attn_fwd_plan(plan, q, k, v, w.alpha, w.inv_n, out)
        torch.cuda.synchronize()
        st, site = binding.hstu_last_status()
        assert st == binding.HSTU_ERR_TIMEOUT
        assert site > 0
    finally:
        binding.hstu_set_debug_flags(0)
        binding.hstu_set_wait_timeout_ns(0)
    # the context is still usable and a normal launch is correct
    out = parity.run_plan(w, q, k, v)
    assert binding.hstu_last_status() == (binding.HSTU_OK, 0)
    assert torch.isfinite(out.float()).all()
    binding.hstu_plan_destroy(plan)
