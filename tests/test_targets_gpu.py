"""GPU parity of the candidate (M-FALCON) mask against the fp64 oracle.

HSTU paper section 3.4 and Appendix H, Algorithm 1: the last num_targets[b]
tokens of sequence b see the history and themselves only.  Every output
element must satisfy the parity bound of tests/parity.py against
oracle.reference.hstu_fwd(..., num_targets=...).
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


# lengths with the candidate count of each: the history ends inside a key
# block, on a block boundary, before the first block ends, not at all (all
# candidates, in one block and over several: each query block then walks
# its diagonal block alone), candidates spanning several query blocks, no
# candidates
CASES = [(300, 100), (513, 128), (256, 1), (700, 333), (90, 90), (129, 0), (0, 0), (1, 1),
         (640, 500), (385, 2), (300, 300), (384, 384)]


def _draw(w, seed):
    q, k, v = workloads.draw_qkv(w, seed=seed)
    return (q, k, v), parity.to_device(q, k, v)


def _check(w, nt, q, k, v, out):
    ref = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n, num_targets=nt)
    got = out.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    r = parity.ratio(got, ref, rms)
    assert np.all(np.isfinite(got))
    assert r.max() <= 1.0, f"worst err/tol {r.max():.3f} at {np.unravel_index(r.argmax(), r.shape)}"


@pytest.mark.parametrize("d", [32, 64, 128])
def test_candidates_full_parity(d):
    lengths = [n for n, _ in CASES]
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    w = workloads.custom(lengths, heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=400 + d)
    out = torch.empty_like(qd)
    plan = binding.hstu_plan_create_targets(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen)
    try:
        binding.hstu_attn_fwd_plan(plan, qd, kd, vd, w.alpha, w.inv_n, out)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    _check(w, nt, q, k, v, out)


def test_candidates_one_call_equals_plan_and_zero_candidates_equal_causal():
    lengths = [n for n, _ in CASES]
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    w = workloads.custom(lengths, heads=3, d=64)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=450)
    a = torch.empty_like(qd)
    binding.hstu_attn_fwd_targets(qd, kd, vd, w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                  w.alpha, w.inv_n, a)
    plan = binding.hstu_plan_create_targets(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen)
    b = torch.empty_like(qd)
    try:
        binding.hstu_attn_fwd_plan(plan, qd, kd, vd, w.alpha, w.inv_n, b)
        torch.cuda.synchronize()
        assert np.array_equal(binding.hstu_plan_item_hist(plan),
                              binding.hstu_worklist_build_targets(w.offsets, nt, w.heads)[1])
    finally:
        binding.hstu_plan_destroy(plan)
    assert torch.equal(a, b)
    # no candidates: bit-identical to the causal entry point
    z = torch.empty_like(qd)
    binding.hstu_attn_fwd_targets(qd, kd, vd, w.offsets, np.zeros(w.batch, np.int32), w.batch,
                                  w.heads, w.d, w.max_seqlen, w.alpha, w.inv_n, z)
    c = torch.empty_like(qd)
    binding.hstu_attn_fwd(qd, kd, vd, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                          w.inv_n, c)
    torch.cuda.synchronize()
    assert torch.equal(z, c)
    parity.assert_device_ok()


def test_candidates_match_separate_causal_passes_on_the_gpu():
    # Appendix H's identity on the GPU path itself: a candidate's row equals
    # the last row of a causal pass over history + that candidate
    hist, bm, heads, d = 300, 5, 2, 64
    w = workloads.custom([hist + bm], heads=heads, d=d)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=460)
    out = torch.empty_like(qd)
    binding.hstu_attn_fwd_targets(qd, kd, vd, w.offsets, [bm], 1, heads, d, w.max_seqlen, w.alpha,
                                  w.inv_n, out)
    for c in range(bm):
        idx = torch.as_tensor(list(range(hist)) + [hist + c], device="cuda")
        sub = torch.empty((hist + 1, heads, d), dtype=qd.dtype, device="cuda")
        binding.hstu_attn_fwd(qd[idx].contiguous(), kd[idx].contiguous(), vd[idx].contiguous(),
                              [0, hist + 1], 1, heads, d, hist + 1, w.alpha, w.inv_n, sub)
        torch.cuda.synchronize()
        a = out[hist + c].float().cpu().numpy()
        b = sub[hist].float().cpu().numpy()
        ref = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n, num_targets=[bm])[hist + c]
        scale = np.abs(ref).max()
        # both GPU results are within parity of the same oracle row
        assert np.abs(a - ref).max() <= 1e-2 * scale and np.abs(b - ref).max() <= 1e-2 * scale
    parity.assert_device_ok()


def test_candidate_workload_sampled():
    w, nt = workloads.candidate_workload()
    (q, k, v), (qd, kd, vd) = _draw(w, seed=470)
    out = torch.empty_like(qd)
    plan = binding.hstu_plan_create_targets(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen)
    try:
        binding.hstu_attn_fwd_plan(plan, qd, kd, vd, w.alpha, w.inv_n, out)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    rt, rh, nu = parity.sample_rows(w, 256, seed=2)
    # add candidate rows of several sequences
    off = w.offsets.astype(np.int64)
    extra = []
    for b in range(0, w.batch, max(1, w.batch // 8)):
        hist = int(w.lengths[b]) - int(nt[b])
        extra += [off[b] + hist, off[b] + int(w.lengths[b]) - 1]
    rt = np.concatenate([rt, np.array(extra, np.int64)])
    rh = np.concatenate([rh, np.zeros(len(extra), np.int64)])
    ref = reference.hstu_rows(q, k, v, w.offsets, w.alpha, w.inv_n, rt, rh, num_targets=nt)
    got = out[torch.as_tensor(rt, device="cuda"), torch.as_tensor(rh, device="cuda")]
    got = got.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref[:nu] ** 2)))
    assert np.all(np.isfinite(got))
    assert parity.ratio(got, ref, rms).max() <= 1.0
