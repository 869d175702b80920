"""GPU: the backward's transposed form (d <= 64 without the bias).

Where d <= 64 and there is no bias, the backward recomputes S^T = K Q^T with
the keys on the TMEM lanes: P^T and dS^T feed dV and dK from TMEM and dS^T
goes to shared memory for dQ (hstu_bwd_t.cuh).  The other backward GPU tests
run it against the fp64 oracle through the default entry points; these add:
agreement with the row form (HSTU_DEBUG_BWD_ROWS) on ragged lengths, with
and without candidates; many short sequences and sequences ending on block
edges, every element against the oracle; isolation from non-finite values
in the next sequence (rows past a sequence are zeroed before the products
read them); and the bounded give-up path.
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


def _inputs(w, seed, dscale=1.0):
    q, k, v = workloads.draw_qkv(w, seed=seed)
    rng = np.random.default_rng(seed + 1)
    do = workloads.bf16_round((dscale * rng.standard_normal(q.shape)).astype(np.float32))
    return (q, k, v, do), tuple(t.to("cuda").contiguous() for t in (q, k, v, do))


def _bwd(w, dev, nt=None):
    qd, kd, vd, dod = dev
    g = [torch.empty_like(qd) for _ in range(3)]
    if nt is None:
        binding.hstu_attn_bwd(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                              w.inv_n, *g)
    else:
        binding.hstu_attn_bwd_ex(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen,
                                 w.alpha, w.inv_n, *g, num_targets=nt)
    torch.cuda.synchronize()
    parity.assert_device_ok()
    return g


def _check(got, ref, name):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    worst = float(parity.ratio(g, ref, rms).max()) if ref.size else 0.0
    assert worst <= 1.0, f"{name}: worst err/tol {worst:.3f}"
    return worst


EDGE_LENGTHS = [1, 127, 128, 129, 255, 256, 257, 383, 384, 385, 0, 2, 640]


@pytest.mark.parametrize("d", [32, 64])
def test_bwd_t_block_edges_full(d):
    w = workloads.custom(EDGE_LENGTHS, heads=2, d=d)
    host, dev = _inputs(w, seed=900 + d)
    got = _bwd(w, dev)
    ref = reference.hstu_bwd(*host, w.offsets, w.alpha, w.inv_n)
    for gt, rf, name in zip(got, ref, ("dq", "dk", "dv")):
        _check(gt, rf, name)


def test_bwd_t_many_short_sequences_full():
    rng = np.random.default_rng(910)
    lengths = rng.integers(0, 400, size=90)
    lengths[::7] = 1
    lengths[::11] = 0
    w = workloads.custom(lengths, heads=2, d=64)
    host, dev = _inputs(w, seed=911)
    got = _bwd(w, dev)
    ref = reference.hstu_bwd(*host, w.offsets, w.alpha, w.inv_n)
    for gt, rf, name in zip(got, ref, ("dq", "dk", "dv")):
        _check(gt, rf, name)


@pytest.mark.parametrize("with_targets", [False, True])
def test_bwd_t_agrees_with_row_form(with_targets):
    w = workloads.custom([900, 300, 129, 1000, 1], heads=2, d=64)
    nt = np.array([200, 0, 129, 64, 1], dtype=np.int32) if with_targets else None
    host, dev = _inputs(w, seed=920)
    a = _bwd(w, dev, nt)
    try:
        binding.hstu_set_debug_flags(binding.HSTU_DEBUG_BWD_ROWS)
        b = _bwd(w, dev, nt)
    finally:
        binding.hstu_set_debug_flags(0)
    ref = reference.hstu_bwd(*host, w.offsets, w.alpha, w.inv_n, num_targets=nt)
    for x, y, rf, name in zip(a, b, ref, ("dq", "dk", "dv")):
        _check(x, rf, name)
        _check(y, rf, name + " (rows)")
        diff = (x.float() - y.float()).abs().max().item()
        assert diff <= 2e-2 * max(y.float().abs().max().item(), 1e-30), name


def test_bwd_t_nonfinite_values_in_next_sequence_do_not_leak():
    # Sequence 0 ends inside a 128-row block whose tail holds sequence 1's
    # rows; make those rows infinite / NaN: the earlier sequences' dK and dV
    # must not change, bit for bit (each comes from one CTA), nor their dQ
    # beyond the order of its fp32 additions.
    w = workloads.custom([200, 100, 330, 60], heads=2, d=64)
    _, (qd, kd, vd, dod) = _inputs(w, seed=930)
    base = _bwd(w, (qd, kd, vd, dod))
    for s0, s1 in ((200, 300), (630, 690)):
        q2, k2, v2, do2 = (t.clone() for t in (qd, kd, vd, dod))
        q2[s0:s1] = float("inf")
        k2[s0:s1] = float("-inf")
        v2[s0:s1] = float("nan")
        do2[s0:s1] = float("inf")
        got = _bwd(w, (q2, k2, v2, do2))
        assert torch.isfinite(got[0][:s0].float()).all(), s0
        dq_diff = (got[0][:s0].float() - base[0][:s0].float()).abs().max().item()
        assert dq_diff <= 1e-2 * base[0][:s0].float().abs().max().item(), s0
        for x, y, name in zip(got[1:], base[1:], ("dk", "dv")):
            assert torch.equal(x[:s0], y[:s0]), (name, s0)


def test_bwd_t_wait_limit_gives_timeout_status_and_context_survives():
    w = workloads.custom([700, 300, 5], heads=2, d=64)
    host, dev = _inputs(w, seed=940)
    binding.hstu_last_status()
    try:
        binding.hstu_set_wait_timeout_ns(1_000_000)
        binding.hstu_set_debug_flags(binding.HSTU_DEBUG_UNSIGNALLED_WAIT)
        qd, kd, vd, dod = dev
        g = [torch.zeros_like(qd) for _ in range(3)]
        binding.hstu_attn_bwd(qd, kd, vd, dod, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                              w.inv_n, *g)
        torch.cuda.synchronize()
        st, site = binding.hstu_last_status()
        assert st == binding.HSTU_ERR_TIMEOUT and site > 0
    finally:
        binding.hstu_set_debug_flags(0)
        binding.hstu_set_wait_timeout_ns(0)
    got = _bwd(w, dev)
    assert binding.hstu_last_status() == (binding.HSTU_OK, 0)
    ref = reference.hstu_bwd(*host, w.offsets, w.alpha, w.inv_n)
    for gt, rf, name in zip(got, ref, ("dq", "dk", "dv")):
        _check(gt, rf, name)
