"""GPU parity of the candidates-only plan (M-FALCON's cached history).

HSTU paper section 3.4: the history's keys and values serve every batch of
candidates, and only the candidates' outputs are wanted.  A plan made with
HSTU_PLAN_CANDIDATES_ONLY computes the query blocks that hold candidate
rows.  Checked against oracle.reference.hstu_fwd(..., num_targets=...)
with the bound of tests/parity.py:
* every candidate row;
* the history rows that share a block with the first candidates (the same
  values as the full pass);
* every other history row of out keeps its previous contents (a sentinel).
"""
import numpy as np
import pytest
import torch

from hstu_jagged_attention_gb300 import binding, build, workloads
from oracle import reference
from tests import parity

pytestmark = pytest.mark.gpu

SENTINEL = 3.0  # exact in bf16; no attention output of these inputs is this value


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.hstu_set_wait_timeout_ns(0)
    yield
    parity.assert_device_ok()


# (length, candidates): history multiple of 128, one candidate, all
# candidates, none, candidates spanning several blocks
CASES = [(300, 100), (513, 128), (256, 1), (700, 333), (90, 90), (129, 0), (0, 0), (1, 1),
         (640, 500), (385, 2), (384, 128), (1000, 999)]


def _rows_computed(w, nt):
    """Token mask of the rows the plan computes: rows of query blocks that
    hold a candidate row."""
    comp = np.zeros(w.total, dtype=bool)
    for b in range(w.batch):
        s0, n = int(w.offsets[b]), int(w.lengths[b])
        hist = n - int(nt[b])
        if hist >= n:
            continue
        comp[s0 + (hist // 128) * 128: s0 + n] = True
    return comp


def _run(w, nt, q, k, v, rab=None):
    qd, kd, vd = parity.to_device(q, k, v)
    out = torch.full_like(qd, SENTINEL)
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_CANDIDATES_ONLY)
    try:
        binding.hstu_attn_fwd_plan_ex(plan, qd, kd, vd, w.alpha, w.inv_n, out, rab=rab)
        torch.cuda.synchronize()
    finally:
        binding.hstu_plan_destroy(plan)
    parity.assert_device_ok()
    return out.float().cpu().numpy().astype(np.float64)


def _check(got, ref, comp):
    rows = got[comp]
    want = ref[comp]
    assert np.all(np.isfinite(rows))
    rms = float(np.sqrt(np.mean(want ** 2))) if want.size else 0.0
    r = parity.ratio(rows, want, rms)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= 1.0, f"worst err/tol {worst:.3f}"
    assert np.all(got[~comp] == SENTINEL), "a history row outside the candidates' blocks was written"


@pytest.mark.parametrize("d", [32, 64, 128])
def test_candidates_only_parity(d):
    w = workloads.custom([n for n, _ in CASES], heads=2, d=d, sigma=1.0 if d < 128 else 0.5)
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    q, k, v = workloads.draw_qkv(w, seed=1400 + d)
    got = _run(w, nt, q, k, v)
    ref = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n, num_targets=nt)
    comp = _rows_computed(w, nt)
    assert comp.any() and (~comp).any()
    _check(got, ref, comp)


def test_candidates_only_with_the_bias():
    w = workloads.custom([n for n, _ in CASES], heads=2, d=64)
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    q, k, v = workloads.draw_qkv(w, seed=1450)
    ts, pos, time = workloads.draw_rab(w, seed=1451, backwards=0.1)
    rab_d = tuple(torch.from_numpy(x).cuda() for x in (ts, pos, time))
    got = _run(w, nt, q, k, v, rab=rab_d)
    ref = reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n, num_targets=nt, rab=(ts, pos, time))
    _check(got, ref, _rows_computed(w, nt))


def test_candidates_only_equals_the_full_candidate_pass_on_its_rows():
    # same kernel, same per-item work: the rows it computes are bit-identical
    w = workloads.custom([n for n, _ in CASES], heads=2, d=64)
    nt = np.array([c for _, c in CASES], dtype=np.int32)
    q, k, v = workloads.draw_qkv(w, seed=1460)
    got = _run(w, nt, q, k, v)
    qd, kd, vd = parity.to_device(q, k, v)
    full = torch.empty_like(qd)
    binding.hstu_attn_fwd_targets(qd, kd, vd, w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                  w.alpha, w.inv_n, full)
    torch.cuda.synchronize()
    comp = _rows_computed(w, nt)
    assert np.array_equal(got[comp], full.float().cpu().numpy().astype(np.float64)[comp])


def test_candidate_workload_candidates_only_sampled():
    # full size: 32 histories of 2048..8192 tokens, 1024 candidates each
    w, nt = workloads.candidate_workload()
    q, k, v = workloads.draw_qkv(w)
    got = _run(w, nt, q, k, v)
    rng = np.random.default_rng(1470)
    off = w.offsets.astype(np.int64)
    cand_t = np.concatenate([np.arange(off[b + 1] - nt[b], off[b + 1]) for b in range(w.batch)])
    rt = rng.choice(cand_t, size=256, replace=False)
    rh = rng.integers(0, w.heads, size=256)
    ref = reference.hstu_rows(q, k, v, w.offsets, w.alpha, w.inv_n, rt, rh, num_targets=nt)
    rows = got[rt, rh]
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert parity.ratio(rows, ref, rms).max() <= 1.0
    comp = _rows_computed(w, nt)
    hist_t = np.flatnonzero(~comp)
    assert np.all(got[hist_t[::97]] == SENTINEL)
