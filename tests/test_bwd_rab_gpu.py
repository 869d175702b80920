"""GPU parity of the backward with the relative attention bias rab_{p,t}.

HSTU paper section 3 (rab_{p,t} inside the nonlinearity) and Appendix G
(the bias's construction fused into the attention, forward and backward).
dq, dk, dv and the tables' gradients dpos, dtime of sum(out * dout) are
checked element by element against oracle.reference.hstu_bwd(...,
rab=..., table_grads=True) with the bound of tests/parity.py, each with its
own rms.
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


def _inputs(w, seed, npos=32, ntime=32):
    q, k, v = workloads.draw_qkv(w, seed=seed)
    rng = np.random.default_rng(seed + 1)
    do = workloads.bf16_round(rng.standard_normal(q.shape).astype(np.float32))
    ts, pos, time = workloads.draw_rab(w, seed=seed + 2, backwards=0.1)
    return q, k, v, do, (ts, pos[:npos].copy(), time[:ntime].copy())


def _dev(q, k, v, do, rab):
    qd, kd, vd, dod = (t.to("cuda").contiguous() for t in (q, k, v, do))
    rd = tuple(torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in rab)
    return qd, kd, vd, dod, rd


def _run(w, q, k, v, do, rab):
    qd, kd, vd, dod, rd = _dev(q, k, v, do, rab)
    g = [torch.empty_like(qd) for _ in range(3)]
    dpos = torch.full((rab[1].size,), float("nan"), device="cuda")
    dtime = torch.full((rab[2].size,), float("nan"), device="cuda")
    binding.hstu_attn_bwd_ex(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen,
                             w.alpha, w.inv_n, *g, rab=rd, dpos=dpos, dtime=dtime)
    torch.cuda.synchronize()
    parity.assert_device_ok()
    return g + [dpos, dtime]


def _check(got, ref, name):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    r = parity.ratio(g, ref, rms)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f} at {np.unravel_index(r.argmax(), r.shape)}"


NAMES = ("dq", "dk", "dv", "dpos", "dtime")


@pytest.mark.parametrize("d,npos,ntime", [(32, 32, 32), (64, 32, 32), (64, 5, 17), (128, 32, 1),
                                          (128, 12, 32)])
def test_bwd_rab_full_parity(d, npos, ntime):
    w = workloads.custom(LENGTHS, heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    q, k, v, do, rab = _inputs(w, 900 + d + npos, npos, ntime)
    got = _run(w, q, k, v, do, rab)
    ref = reference.hstu_bwd(q, k, v, do, w.offsets, w.alpha, w.inv_n, rab=rab, table_grads=True)
    for gt, rf, name in zip(got, ref, NAMES):
        _check(gt, rf, name)


def test_bwd_rab_long_sequences():
    w = workloads.custom([2048, 1500], heads=2, d=64)
    q, k, v, do, rab = _inputs(w, 950)
    got = _run(w, q, k, v, do, rab)
    ref = reference.hstu_bwd(q, k, v, do, w.offsets, w.alpha, w.inv_n, rab=rab, table_grads=True)
    for gt, rf, name in zip(got, ref, NAMES):
        _check(gt, rf, name)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_zero_tables_give_the_plain_dk_dv_bit_for_bit(d):
    # a zero bias adds exactly zero to every score: dk and dv (one CTA's
    # sums each, in the same order) equal the plain kernel's in the row form,
    # which the bias runs in (HSTU_DEBUG_BWD_ROWS makes the plain call run
    # it too), and the default plain form (transposed for d <= 64) within
    # the tolerance; dq sums parts with atomics in an order that may differ
    w = workloads.custom([700, 1, 129, 256], heads=2, d=d)
    q, k, v, do, rab = _inputs(w, 960 + d)
    rab = (rab[0], np.zeros_like(rab[1]), np.zeros_like(rab[2]))
    qd, kd, vd, dod, _ = _dev(q, k, v, do, rab)

    def plain_bwd():
        g = [torch.empty_like(qd) for _ in range(3)]
        binding.hstu_attn_bwd(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                              w.inv_n, *g)
        torch.cuda.synchronize()
        return g

    got = _run(w, q, k, v, do, rab)
    try:
        binding.hstu_set_debug_flags(binding.HSTU_DEBUG_BWD_ROWS)
        rows = plain_bwd()
    finally:
        binding.hstu_set_debug_flags(0)
    default = plain_bwd()
    assert torch.equal(got[1], rows[1]) and torch.equal(got[2], rows[2])
    for x, y in ((got[0], rows[0]), (got[0], default[0]), (got[1], default[1]), (got[2], default[2])):
        assert (x.float() - y.float()).abs().max().item() <= 1e-2 * y.float().abs().max().item()


def test_bwd_rab_plan_equals_one_shot():
    w = workloads.custom(LENGTHS, heads=2, d=64)
    q, k, v, do, rab = _inputs(w, 970, 20, 29)
    a = _run(w, q, k, v, do, rab)
    qd, kd, vd, dod, rd = _dev(q, k, v, do, rab)
    g = [torch.empty_like(qd) for _ in range(3)]
    dpos, dtime = torch.empty(20, device="cuda"), torch.empty(29, device="cuda")
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)
    try:
        for _ in range(2):  # the accumulators restart on every call
            binding.hstu_attn_bwd_plan_ex(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g, rab=rd,
                                          dpos=dpos, dtime=dtime)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    assert torch.equal(g[1], a[1]) and torch.equal(g[2], a[2])
    for x, y in ((g[0], a[0]), (dpos, a[3]), (dtime, a[4])):
        assert (x.float() - y.float()).abs().max().item() <= 1e-3 * y.float().abs().max().item() + 1e-6


def test_bwd_rab_empty_batch_zeroes_the_table_gradients():
    w = workloads.custom([0, 0], heads=2, d=64)
    dpos = torch.full((32,), 7.0, device="cuda")
    dtime = torch.full((9,), 7.0, device="cuda")
    z = torch.zeros(8, 2, 64, dtype=torch.bfloat16, device="cuda")
    ts = torch.zeros(8, dtype=torch.int32, device="cuda")
    tab = torch.zeros(32, device="cuda")
    binding.hstu_attn_bwd_ex(z, z, z, z, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                             w.inv_n, z, z, z, rab=(ts, tab, tab[:9]), dpos=dpos, dtime=dtime)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dpos).item() == 0 and torch.count_nonzero(dtime).item() == 0


def test_bwd_rab_dense_workload_sampled():
    # full size, in the launch configuration the benchmark times (a plan)
    w = workloads.workload("dense")
    q, k, v = workloads.draw_qkv(w)
    rng = np.random.default_rng(4000 + w.index)
    do = workloads.bf16_round(rng.standard_normal(q.shape).astype(np.float32))
    rab = workloads.draw_rab(w)
    qd, kd, vd, dod, rd = _dev(q, k, v, do, rab)
    g = [torch.empty_like(qd) for _ in range(3)]
    dpos, dtime = torch.empty(32, device="cuda"), torch.empty(32, device="cuda")
    plan = binding.hstu_plan_create_ex(w.offsets, None, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)
    try:
        binding.hstu_attn_bwd_plan_ex(plan, qd, kd, vd, dod, w.alpha, w.inv_n, *g, rab=rd,
                                      dpos=dpos, dtime=dtime)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    rt, rh, nu = parity.sample_rows(w, 192, seed=8)
    refs = reference.hstu_bwd_rows(q, k, v, do, w.offsets, w.alpha, w.inv_n, rt, rh, rab=rab)
    idx_t, idx_h = torch.as_tensor(rt, device="cuda"), torch.as_tensor(rh, device="cuda")
    for name, gt, rf in zip(("dq", "dk", "dv"), g, refs):
        got = gt[idx_t, idx_h].float().cpu().numpy().astype(np.float64)
        rms = float(np.sqrt(np.mean(rf[:nu] ** 2)))
        assert np.all(np.isfinite(got)), name
        worst = parity.ratio(got, rf, rms).max()
        assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f}"
    # every kept pair adds its ds to one position and one time bucket: the
    # two tables' gradients have the same total
    sp, st = dpos.double().sum().item(), dtime.double().sum().item()
    scale = dpos.double().abs().sum().item() + dtime.double().abs().sum().item()
    assert np.isfinite(sp) and abs(sp - st) <= 1e-4 * scale
