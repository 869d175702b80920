"""GPU parity of the relative attention bias rab_{p,t} against the fp64 oracle.

HSTU paper section 3 (rab_{p,t}) and section 3.4 (M-FALCON: candidates sit
at the history's end).  Every output element must satisfy the parity bound
of tests/parity.py against oracle.reference.hstu_fwd(..., rab=...).
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


CASES = [(300, 100), (513, 128), (256, 1), (700, 333), (90, 90), (129, 0), (0, 0), (1, 1),
         (640, 500), (385, 2)]


def _dev_rab(ts, pos, time):
    return (torch.from_numpy(ts).cuda(), torch.from_numpy(pos).cuda(), torch.from_numpy(time).cuda())


def _check(ref, y):
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    r = parity.ratio(got, ref, rms)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= 1.0, f"worst err/tol {worst:.3f} at {np.unravel_index(r.argmax(), r.shape)}"


@pytest.mark.parametrize("d,targets", [(32, False), (32, True), (64, False), (64, True),
                                       (128, False), (128, True)])
def test_rab_full_parity(d, targets):
    lengths = [n for n, _ in CASES]
    nt = np.array([c for _, c in CASES], dtype=np.int32) if targets else None
    w = workloads.custom(lengths, heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    q, k, v = workloads.draw_qkv(w, seed=700 + d)
    ts, pos, time = workloads.draw_rab(w, seed=710 + d, backwards=0.1)
    rng = np.random.default_rng(d)
    pos, time = pos[:int(rng.integers(1, 33))], time[:int(rng.integers(1, 33))]
    qd, kd, vd = parity.to_device(q, k, v)
    out = torch.empty_like(qd)
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen, 0)
    try:
        binding.hstu_attn_fwd_plan_ex(plan, qd, kd, vd, w.alpha, w.inv_n, out,
                                      rab=_dev_rab(ts, pos, time))
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    ref = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n, num_targets=nt, rab=(ts, pos, time))
    _check(ref, out)


def test_zero_tables_give_the_plain_kernel_bit_for_bit():
    w = workloads.custom([700, 1, 129, 256], heads=2, d=64)
    q, k, v = workloads.draw_qkv(w, seed=720)
    ts, _, _ = workloads.draw_rab(w, seed=721)
    qd, kd, vd = parity.to_device(q, k, v)
    a, b = torch.empty_like(qd), torch.empty_like(qd)
    z = np.zeros(32, np.float32)
    binding.hstu_attn_fwd_ex(qd, kd, vd, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                             w.inv_n, a, rab=_dev_rab(ts, z, z))
    binding.hstu_attn_fwd(qd, kd, vd, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                          w.inv_n, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_every_option_at_once_one_shot_equals_plan():
    lengths = [n for n, _ in CASES]
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    w = workloads.custom(lengths, heads=3, d=64)
    q, k, v = workloads.draw_qkv(w, seed=730)
    u, g, b = workloads.draw_norm_gate(w, seed=731)
    ts, pos, time = workloads.draw_rab(w, seed=732)
    qd, kd, vd = parity.to_device(q, k, v)
    ud, gd, bd = u.cuda(), torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda()
    rab = _dev_rab(ts, pos, time)
    ng = (ud, gd, bd, workloads.NORM_EPS)
    y1, y2 = torch.empty_like(qd), torch.empty_like(qd)
    binding.hstu_attn_fwd_ex(qd, kd, vd, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                             w.inv_n, y1, num_targets=nt, rab=rab, norm_gate=ng)
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_NORM_GATE)
    try:
        binding.hstu_attn_fwd_plan_ex(plan, qd, kd, vd, w.alpha, w.inv_n, y2, rab=rab, norm_gate=ng)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    assert torch.equal(y1, y2)
    ref = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, workloads.NORM_EPS, w.offsets, w.alpha,
                                       w.inv_n, num_targets=nt, rab=(ts, pos, time))
    _check(ref, y1)
    parity.assert_device_ok()


def test_candidates_match_separate_causal_passes_with_bias_on_the_gpu():
    hist, bm, heads, d = 300, 4, 2, 64
    w = workloads.custom([hist + bm], heads=heads, d=d)
    q, k, v = workloads.draw_qkv(w, seed=740)
    ts, pos, time = workloads.draw_rab(w, seed=741)
    qd, kd, vd = parity.to_device(q, k, v)
    out = torch.empty_like(qd)
    binding.hstu_attn_fwd_ex(qd, kd, vd, w.offsets, 1, heads, d, w.max_seqlen, w.alpha, w.inv_n, out,
                             num_targets=[bm], rab=_dev_rab(ts, pos, time))
    ref = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n, num_targets=[bm],
                             rab=(ts, pos, time))
    for c in range(bm):
        idx = list(range(hist)) + [hist + c]
        sub = torch.empty((hist + 1, heads, d), dtype=qd.dtype, device="cuda")
        binding.hstu_attn_fwd_ex(qd[idx].contiguous(), kd[idx].contiguous(), vd[idx].contiguous(),
                                 [0, hist + 1], 1, heads, d, hist + 1, w.alpha, w.inv_n, sub,
                                 rab=_dev_rab(np.ascontiguousarray(ts[idx]), pos, time))
        torch.cuda.synchronize()
        scale = np.abs(ref[hist + c]).max()
        a = out[hist + c].float().cpu().numpy()
        b = sub[hist].float().cpu().numpy()
        assert np.abs(a - ref[hist + c]).max() <= 1e-2 * scale
        assert np.abs(b - ref[hist + c]).max() <= 1e-2 * scale
    parity.assert_device_ok()


def test_dense_workload_sampled():
    w = workloads.workload("dense")
    q, k, v = workloads.draw_qkv(w)
    ts, pos, time = workloads.draw_rab(w)
    qd, kd, vd = parity.to_device(q, k, v)
    out = torch.empty_like(qd)
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen, 0)
    try:
        binding.hstu_attn_fwd_plan_ex(plan, qd, kd, vd, w.alpha, w.inv_n, out,
                                      rab=_dev_rab(ts, pos, time))
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    rt, rh, nu = parity.sample_rows(w, 256, seed=5)
    ref = reference.hstu_rows(q, k, v, w.offsets, w.alpha, w.inv_n, rt, rh, rab=(ts, pos, time))
    got = out[torch.as_tensor(rt, device="cuda"), torch.as_tensor(rh, device="cuda")]
    got = got.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref[:nu] ** 2)))
    assert np.all(np.isfinite(got))
    assert parity.ratio(got, ref, rms).max() <= 1.0
