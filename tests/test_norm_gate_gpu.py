"""GPU parity of the output stage y = Norm(A V) (.) U against the fp64 oracle.

HSTU paper section 3 and section 3.1: a layer norm over each token's
heads * d attention outputs, affine gamma and beta, times U.  Every element
of y must satisfy the parity bound of tests/parity.py against
oracle.reference.hstu_fwd_norm_gate on the same bf16 inputs.
"""
import numpy as np
import pytest
import torch

from hstu_jagged_attention_gb300 import binding, build, workloads
from oracle import reference
from tests import parity

pytestmark = pytest.mark.gpu

NG = binding.HSTU_PLAN_NORM_GATE


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.hstu_set_wait_timeout_ns(0)
    yield
    parity.assert_device_ok()


# lengths with candidate counts: ragged tails, block boundaries, empties,
# single tokens, all-candidate sequences
CASES = [(300, 100), (513, 128), (256, 1), (700, 333), (90, 90), (129, 0), (0, 0), (1, 1),
         (640, 500), (385, 2)]


def _inputs(w, seed):
    q, k, v = workloads.draw_qkv(w, seed=seed)
    u, g, b = workloads.draw_norm_gate(w, seed=seed + 1)
    dev = [t.to("cuda").contiguous() for t in (q, k, v, u)]
    gd, bd = torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda()
    return (q, k, v, u, g, b), (*dev, gd, bd)


def _run_plan(w, nt, dev, eps, y=None, plan=None):
    qd, kd, vd, ud, gd, bd = dev
    y = torch.empty_like(qd) if y is None else y
    own = plan is None
    if own:
        plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen, NG)
    try:
        binding.hstu_attn_fwd_norm_gate_plan(plan, qd, kd, vd, ud, gd, bd, eps, w.alpha, w.inv_n, y)
        torch.cuda.synchronize()
    finally:
        if own:
            binding.hstu_plan_destroy(plan)
    return y


def _check(ref, y):
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    r = parity.ratio(got, ref, rms)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= 1.0, f"worst err/tol {worst:.3f} at {np.unravel_index(r.argmax(), r.shape)}"
    return worst


@pytest.mark.parametrize("d,heads,targets", [(32, 1, False), (32, 3, True), (64, 3, False),
                                             (64, 4, True), (128, 2, False), (128, 2, True)])
def test_norm_gate_full_parity(d, heads, targets):
    lengths = [n for n, _ in CASES]
    nt = np.array([c for _, c in CASES], dtype=np.int32) if targets else None
    w = workloads.custom(lengths, heads=heads, d=d, sigma=1.0 if d < 128 else 0.5)
    (q, k, v, u, g, b), dev = _inputs(w, seed=600 + d + heads)
    eps = workloads.NORM_EPS
    y = _run_plan(w, nt, dev, eps)
    parity.assert_device_ok()
    ref = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, eps, w.offsets, w.alpha, w.inv_n,
                                       num_targets=nt)
    _check(ref, y)


def test_norm_gate_without_eps_and_unit_inv_n():
    # eps = 0: pure standardisation of every row (no row here has zero variance)
    w = workloads.custom([333, 1, 129, 700], heads=2, d=64, inv_n=1.0)
    (q, k, v, u, g, b), dev = _inputs(w, seed=650)
    y = _run_plan(w, None, dev, 0.0)
    ref = reference.hstu_fwd_norm_gate(q, k, v, u, g, b, 0.0, w.offsets, w.alpha, w.inv_n)
    _check(ref, y)


def test_one_shot_equals_plan_and_the_plan_serves_plain_attention():
    lengths = [n for n, _ in CASES]
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    w = workloads.custom(lengths, heads=3, d=64)
    (q, k, v, u, g, b), dev = _inputs(w, seed=660)
    qd, kd, vd, ud, gd, bd = dev
    eps = workloads.NORM_EPS
    a = _run_plan(w, nt, dev, eps)
    c = torch.empty_like(qd)
    binding.hstu_attn_fwd_norm_gate(qd, kd, vd, ud, gd, bd, eps, w.offsets, nt, w.batch, w.heads,
                                    w.d, w.max_seqlen, w.alpha, w.inv_n, c)
    torch.cuda.synchronize()
    assert torch.equal(a, c)
    # a plan with the flag also runs the plain attention, bit for bit
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen, NG)
    try:
        o1 = torch.empty_like(qd)
        binding.hstu_attn_fwd_plan(plan, qd, kd, vd, w.alpha, w.inv_n, o1)
        items, hist = binding.hstu_worklist_build_targets(w.offsets, nt, w.heads)
        assert np.array_equal(binding.hstu_plan_worklist(plan), items)
        assert np.array_equal(binding.hstu_plan_item_hist(plan), hist)
        # the same plan, reused: the scratch slots are rewritten, not accumulated
        y2 = _run_plan(w, nt, dev, eps, plan=plan)
        assert torch.equal(a, y2)
    finally:
        binding.hstu_plan_destroy(plan)
    o2 = torch.empty_like(qd)
    binding.hstu_attn_fwd_targets(qd, kd, vd, w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                  w.alpha, w.inv_n, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    parity.assert_device_ok()


def test_norm_gate_matches_norm_of_the_gpu_attention():
    # the output stage applied (in fp64 on the host) to the GPU's own bf16
    # attention output lands within bf16 rounding of the fused result
    w = workloads.custom([700, 129, 1, 512], heads=4, d=64, inv_n=1.0)
    (q, k, v, u, g, b), dev = _inputs(w, seed=670)
    qd, kd, vd = dev[:3]
    eps = workloads.NORM_EPS
    y = _run_plan(w, None, dev, eps).float().cpu().numpy().astype(np.float64)
    o = torch.empty_like(qd)
    binding.hstu_attn_fwd(qd, kd, vd, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                          w.inv_n, o)
    torch.cuda.synchronize()
    x = o.float().cpu().numpy().astype(np.float64)
    host = reference.norm_gate(x, u, g, b, eps)
    # the host path normalises x rounded to bf16 (|dx| <= 2^-9 |x|), which moves
    # each normalised value by at most 2^-9 (|x| + mean |x|) rstd; both results
    # are then rounded to bf16 once more
    rows = x.reshape(len(x), -1)
    rstd = 1.0 / np.sqrt(rows.var(axis=1) + eps)
    spread = (np.abs(rows) + np.abs(rows).mean(axis=1, keepdims=True)) * rstd[:, None]
    gu = np.abs(g.astype(np.float64))[None, :] * np.abs(u.float().numpy().reshape(len(x), -1))
    rms = float(np.sqrt(np.mean(host ** 2)))
    tol = 2.0 ** -8 * (spread * gu + np.abs(host.reshape(len(x), -1))) + 1e-3 * rms
    assert np.all(np.abs(y - host).reshape(len(x), -1) <= tol)


def test_dense_workload_sampled():
    w = workloads.workload("dense")
    (q, k, v, u, g, b), dev = _inputs(w, seed=680)
    eps = workloads.NORM_EPS
    y = _run_plan(w, None, dev, eps)
    parity.assert_device_ok()
    rng = np.random.default_rng(3)
    off = w.offsets.astype(np.int64)
    rows = list(rng.integers(0, w.total, size=48))
    for bb in (0, w.batch // 2, w.batch - 1):   # first, block-boundary and last tokens
        rows += [off[bb], off[bb] + 127, off[bb] + 128, off[bb + 1] - 1]
    rows = np.array(rows, dtype=np.int64)
    ref = reference.hstu_rows_norm_gate(q, k, v, u, g, b, eps, w.offsets, w.alpha, w.inv_n, rows)
    got = y[torch.as_tensor(rows, device="cuda")].float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref[:48] ** 2)))
    assert np.all(np.isfinite(got))
    assert parity.ratio(got, ref, rms).max() <= 1.0
