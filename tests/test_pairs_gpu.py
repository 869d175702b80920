"""GPU parity of the forward on CTA pairs (two-CTA clusters, d = 64 and 128).

A pair item covers query blocks 2 qp and 2 qp + 1 of one (sequence,
head); the cluster's tensor products run 256 rows over both SMs.  Plans made
with HSTU_PLAN_PAIRS use the pair work list (where it applies; other plans
run one CTA per item), so these tests run the pair kernel on ragged inputs
and on the full dense workload.  Every output element is compared with the
fp64 oracle at the stated tolerance; causality, isolation from non-finite
values of the next sequence, untouched rows past the end, agreement with the
one-CTA path and the bounded give-up path are checked as for that path.
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
    binding.hstu_set_wait_timeout_ns(0)
    yield
    parity.assert_device_ok()


def _draw(w, seed=None):
    q, k, v = workloads.draw_qkv(w, seed)
    return (q, k, v), parity.to_device(q, k, v)


def run_pairs(w, q, k, v, out=None):
    out = torch.empty_like(q) if out is None else out
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_PAIRS)
    try:
        assert binding.hstu_plan_num_pairs(plan) > 0
        binding.hstu_attn_fwd_plan(plan, q, k, v, w.alpha, w.inv_n, out)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    return out


# sequences ending on and around the 128- and 256-row boundaries of pairs:
# a pair whose second block is empty (odd block counts), partial blocks in
# either CTA, a 1-token sequence, an empty one
PAIR_LENGTHS = [1, 127, 128, 129, 255, 256, 257, 383, 384, 385, 511, 512, 513, 0, 700, 2]


@pytest.mark.parametrize("d", [64, 128])
def test_pair_ragged_full(d):
    w = workloads.custom(PAIR_LENGTHS, heads=3, d=d, sigma=1.0 if d < 128 else 0.5)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=80 + d)
    out = run_pairs(w, qd, kd, vd)
    parity.full_check(w, q, k, v, out)
    parity.assert_device_ok()


@pytest.mark.parametrize("d", [64, 128])
def test_pair_many_short_sequences_full(d):
    rng = np.random.default_rng(90 + d)
    lengths = rng.integers(0, 600, size=120)
    lengths[::7] = 1
    lengths[::11] = 0
    w = workloads.custom(lengths, heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=100 + d)
    out = run_pairs(w, qd, kd, vd)
    parity.full_check(w, q, k, v, out)


@pytest.mark.parametrize("d", [64, 128])
def test_pair_path_agrees_with_one_cta_path(d):
    w = workloads.custom([900, 300, 129, 1000], heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=110 + d)
    a = run_pairs(w, qd, kd, vd)
    try:
        binding.hstu_set_debug_flags(binding.HSTU_DEBUG_NO_PAIRS)
        b = run_pairs(w, qd, kd, vd)  # the same plan kind, launched on one CTA per item
    finally:
        binding.hstu_set_debug_flags(0)
    ref = parity.full_check(w, q, k, v, a)
    parity.full_check(w, q, k, v, b)
    diff = (a.float() - b.float()).abs()
    assert diff.max().item() <= 1e-2 * max(b.float().abs().max().item(), 1e-30) + 1e-6, ref


def test_pair_plan_launch_shape():
    # a pair plan launches whole clusters of two CTAs, one CTA per SM at most
    for name in ("dense", "long"):
        w = workloads.workload(name)
        plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                           binding.HSTU_PLAN_PAIRS)
        try:
            assert binding.hstu_plan_num_pairs(plan) > 0, name
            grid, block, smem = binding.hstu_launch_shape(plan)
            assert grid % 2 == 0 and grid <= 152 and block == 512 and smem > 0
        finally:
            binding.hstu_plan_destroy(plan)


def test_pair_full_size_dense_sampled():
    w = workloads.workload("dense")
    (q, k, v), (qd, kd, vd) = _draw(w)
    out = run_pairs(w, qd, kd, vd)
    parity.assert_device_ok()
    parity.sampled_check(w, q, k, v, out, n_random=256, seed=2)


def test_pair_causality_bit_exact():
    # Rows <= i ignore keys and values after i, on pairs as on one CTA.
    w = workloads.custom([700, 300], heads=2, d=64)
    _, (qd, kd, vd) = _draw(w, seed=120)
    base = run_pairs(w, qd, kd, vd)
    for i in (0, 127, 128, 255, 256, 450, 698):
        k2, v2 = kd.clone(), vd.clone()
        k2[i + 1:700] = torch.randn_like(k2[i + 1:700].float()).to(k2.dtype) * 3
        v2[i + 1:700] = torch.randn_like(v2[i + 1:700].float()).to(v2.dtype) * 3
        out = run_pairs(w, qd, k2, v2)
        assert torch.equal(out[: i + 1], base[: i + 1]), i
        assert torch.equal(out[700:], base[700:])


@pytest.mark.parametrize("d", [64, 128])
def test_pair_nonfinite_values_in_next_sequence_do_not_leak(d):
    # The last key block of a sequence reaches into the next sequence; its
    # Inf keys and NaN values must not reach this sequence's rows (both
    # CTAs' V halves are zeroed past the end).
    w = workloads.custom([200, 100, 330, 60], heads=2, d=d)
    _, (qd, kd, vd) = _draw(w, seed=130 + d)
    base = run_pairs(w, qd, kd, vd)
    for s0, s1 in ((200, 300), (630, 690)):
        k2, v2 = kd.clone(), vd.clone()
        k2[s0:s1] = float("inf")
        v2[s0:s1] = float("nan")
        out = run_pairs(w, qd, k2, v2)
        assert torch.equal(out[:s0], base[:s0])


def test_pair_only_valid_rows_written():
    w = workloads.custom([130, 1, 257, 385], heads=2, d=128, sigma=0.5)
    _, (qd, kd, vd) = _draw(w, seed=140)
    canary = torch.full((w.total + 64, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    canary_bits = canary.view(torch.int16).clone()
    out = canary[: w.total]
    run_pairs(w, qd, kd, vd, out=out)
    assert torch.isfinite(out.float()).all()
    assert torch.equal(canary.view(torch.int16)[w.total:], canary_bits[w.total:])


def test_pair_wait_limit_gives_timeout_status_and_context_survives():
    w = workloads.custom([700, 300, 5], heads=2, d=64)
    q, k, v = parity.to_device(*workloads.draw_qkv(w, seed=160))
    binding.hstu_last_status()
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_PAIRS)
    try:
        binding.hstu_set_wait_timeout_ns(1_000_000)
        binding.hstu_set_debug_flags(binding.HSTU_DEBUG_UNSIGNALLED_WAIT)
        out = torch.zeros_like(q)
        binding.hstu_attn_fwd_plan(plan, q, k, v, w.alpha, w.inv_n, out)
        torch.cuda.synchronize()
        st, site = binding.hstu_last_status()
        assert st == binding.HSTU_ERR_TIMEOUT and site > 0
    finally:
        binding.hstu_set_debug_flags(0)
        binding.hstu_set_wait_timeout_ns(0)
        binding.hstu_plan_destroy(plan)
    out = run_pairs(w, q, k, v)
    assert binding.hstu_last_status() == (binding.HSTU_OK, 0)
    assert torch.isfinite(out.float()).all()
