"""The C-ABI library: load, exported symbols, host work list, validation.

These run without a GPU: no call here launches a kernel.  The work list is
compared bit for bit with the oracle's plain-Python enumeration.
"""
import os
import re

import numpy as np
import pytest

from hstu_jagged_attention_gb300 import binding, build, workloads
from oracle import worklist as oracle_worklist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "hstu_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hstu_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert _declared_functions() == binding.exported_symbols()


def test_library_exports_every_declared_symbol():
    L = binding.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {binding.LIB_PATH}").read()
    exported = set(re.findall(r" T (hstu_[a-z_0-9]+)", out))
    assert set(_declared_functions()) <= exported


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5):
        assert binding.hstu_status_string(code)
    assert binding.hstu_status_string(-99) == "unknown status"


@pytest.mark.parametrize("name", workloads.WORKLOAD_NAMES)
def test_worklist_bit_exact_vs_oracle(name):
    w = workloads.workload(name)
    got = binding.hstu_worklist_build(w.offsets, w.heads)
    ref = oracle_worklist.items(w.offsets, w.heads)
    assert got.dtype == np.int32 and got.shape == ref.shape
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("seed", range(20))
def test_worklist_bit_exact_random(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(0, 40))
    lengths = rng.integers(0, 1200, size=nb) * (rng.random(nb) > 0.2)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    heads = int(rng.integers(1, 6))
    got = binding.hstu_worklist_build(off, heads)
    ref = oracle_worklist.items(off, heads)
    assert np.array_equal(got.reshape(-1, 4), ref.reshape(-1, 4))


def test_worklist_hand_cases_through_library():
    from tests.test_oracle_pins import _read_worklist_cases
    for offsets, heads, expect in _read_worklist_cases():
        got = binding.hstu_worklist_build(np.array(offsets, np.int32), heads)
        assert got.tolist() == expect


@pytest.mark.parametrize("offsets", [[1, 5], [0, 5, 3], [0, -1]])
def test_worklist_rejects_bad_offsets(offsets):
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_worklist_build(np.array(offsets, np.int32), 2)
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG


def test_worklist_rejects_bad_heads():
    with pytest.raises(binding.HstuError):
        binding.hstu_worklist_build(np.array([0, 4], np.int32), 0)


@pytest.mark.parametrize("args,code", [
    (dict(offsets=[0, 5, 3], d=64, max_seqlen=10), binding.HSTU_ERR_INVALID_ARG),   # decreasing
    (dict(offsets=[2, 5], d=64, max_seqlen=10), binding.HSTU_ERR_INVALID_ARG),      # off[0] != 0
    (dict(offsets=[0, 50], d=64, max_seqlen=10), binding.HSTU_ERR_INVALID_ARG),     # > max_seqlen
    (dict(offsets=[0, 5], d=96, max_seqlen=10), binding.HSTU_ERR_UNSUPPORTED),      # d
    (dict(offsets=[0, 5], d=64, max_seqlen=-1), binding.HSTU_ERR_INVALID_ARG),
])
def test_plan_create_validation(args, code):
    off = np.array(args["offsets"], np.int32)
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_plan_create(off, len(off) - 1, 2, args["d"], args["max_seqlen"])
    assert e.value.code == code


def test_fwd_validation_before_any_cuda_call():
    # Errors found on the arguments return before anything is enqueued.
    off = np.array([0, 4], np.int32)
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_attn_fwd(16, 16, 16, off, 1, 2, 48, 4, 1.0, 1.0, 16, stream=0)
    assert e.value.code == binding.HSTU_ERR_UNSUPPORTED
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_attn_fwd(16, 16, 16, off, 1, 0, 64, 4, 1.0, 1.0, 16, stream=0)
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG
    # batch == 0 is a no-op that succeeds without touching any pointer
    binding.hstu_attn_fwd(0, 0, 0, np.zeros(1, np.int32), 0, 2, 64, 0, 1.0, 1.0, 0, stream=0)


def test_empty_plan_needs_no_device():
    # all sequences empty: no work items, so no device allocation happens
    p = binding.hstu_plan_create(np.zeros(4, np.int32), 3, 2, 64, 0)
    assert binding.hstu_plan_num_items(p) == 0
    assert binding.hstu_plan_worklist(p).shape == (0, 4)
    binding.hstu_attn_fwd_plan(p, 0, 0, 0, 1.0, 1.0, 0, stream=0)  # no-op
    binding.hstu_plan_destroy(p)


def test_build_flags_target_sm103a():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


# ------------------------------------------------ candidates (M-FALCON mask)
@pytest.mark.parametrize("seed", range(12))
def test_candidate_worklist_bit_exact_random(seed):
    rng = np.random.default_rng(300 + seed)
    nb = int(rng.integers(0, 30))
    lengths = rng.integers(0, 900, size=nb)
    nt = [int(rng.integers(0, n + 1)) if rng.random() < 0.8 else 0 for n in lengths]
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    heads = int(rng.integers(1, 5))
    items, hist = binding.hstu_worklist_build_targets(off, nt, heads)
    ref_items, ref_hist = oracle_worklist.items_targets(off, nt, heads)
    assert np.array_equal(items, ref_items.reshape(-1, 4))
    assert np.array_equal(hist, ref_hist)


def test_candidate_worklist_without_candidates_is_the_causal_one():
    w = workloads.workload("serving")
    items, hist = binding.hstu_worklist_build_targets(w.offsets, np.zeros(w.batch, np.int32), w.heads)
    assert np.array_equal(items, binding.hstu_worklist_build(w.offsets, w.heads))
    assert np.array_equal(hist, items[:, 1])


@pytest.mark.parametrize("nt", [[-1, 0], [0, 4], [6, 0]])
def test_candidate_counts_are_validated(nt):
    off = np.array([0, 5, 8], np.int32)   # lengths 5 and 3
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_worklist_build_targets(off, nt, 1)
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_plan_create_targets(off, nt, 2, 1, 64, 8)
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG


# ------------------------------------------------ output stage Norm(A V) (.) U
def test_norm_gate_validation_before_any_cuda_call():
    off = np.array([0, 4], np.int32)
    bad = [dict(u=0), dict(gamma=8), dict(eps=-1.0), dict(eps=float("nan")), dict(beta=0)]
    for kw in bad:
        args = dict(u=16, gamma=16, beta=16, eps=1e-5, heads=2)
        args.update(kw)
        with pytest.raises(binding.HstuError) as e:
            binding.hstu_attn_fwd_norm_gate(16, 16, 16, args["u"], args["gamma"], args["beta"],
                                            args["eps"], off, None, 1, args["heads"], 64, 4, 1.0,
                                            1.0, 16, stream=0)
        assert e.value.code == binding.HSTU_ERR_INVALID_ARG, kw
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_plan_create_ex(off, None, 1, 2, 64, 4, flags=4)
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG


def test_norm_gate_on_a_plan_without_the_flag_is_rejected():
    # an empty plan needs no device; the flag check comes first
    p = binding.hstu_plan_create(np.zeros(3, np.int32), 2, 2, 64, 0)
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_attn_fwd_norm_gate_plan(p, 0, 0, 0, 0, 0, 0, 1e-5, 1.0, 1.0, 0, stream=0)
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG
    binding.hstu_plan_destroy(p)
    q = binding.hstu_plan_create_ex(np.zeros(3, np.int32), None, 2, 2, 64, 0,
                                    flags=binding.HSTU_PLAN_NORM_GATE)
    binding.hstu_attn_fwd_norm_gate_plan(q, 0, 0, 0, 0, 0, 0, 1e-5, 1.0, 1.0, 0, stream=0)  # no-op
    binding.hstu_plan_destroy(q)


# ------------------------------------------------ relative attention bias
def test_rab_validation_before_any_cuda_call():
    off = np.array([0, 4], np.int32)
    good = dict(ts=16, pos=16, npos=8, time=16, ntime=8)
    bad = [dict(ts=0), dict(pos=0), dict(time=0), dict(ts=18), dict(npos=0), dict(npos=33),
           dict(ntime=0), dict(ntime=40)]
    for kw in bad:
        a = dict(good)
        a.update(kw)
        rab = binding._Rab(a["ts"], a["pos"], a["npos"], a["time"], a["ntime"])
        code = binding.lib().hstu_attn_fwd_ex(16, 16, 16, off.ctypes.data, None, 1, 2, 64, 4,
                                              binding.ctypes.pointer(rab), None, 1.0, 1.0, 16, None)
        assert code == binding.HSTU_ERR_INVALID_ARG, kw


def test_rab_draws_are_in_range():
    w = workloads.workload("dense")
    ts, pos, time = workloads.draw_rab(w)
    assert ts.dtype == np.int32 and ts.shape == (w.total,) and ts.min() >= 0
    assert len(pos) == len(time) == workloads.RAB_BUCKETS
    off = w.offsets
    for b in range(w.batch):
        assert np.all(np.diff(ts[off[b]:off[b + 1]].astype(np.int64)) >= 0)


# ------------------------------------------------ backward work list
@pytest.mark.parametrize("seed", range(8))
def test_bwd_worklist_bit_exact_random(seed):
    rng = np.random.default_rng(900 + seed)
    nb = int(rng.integers(0, 30))
    lengths = rng.integers(0, 900, size=nb)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    heads = int(rng.integers(1, 5))
    got = binding.hstu_worklist_build_bwd(off, heads)
    assert np.array_equal(got, oracle_worklist.items_bwd(off, heads).reshape(-1, 4))


def test_bwd_validation_before_any_cuda_call():
    off = np.array([0, 4], np.int32)
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_attn_bwd(16, 16, 16, 16, off, 1, 2, 48, 4, 1.0, 1.0, 16, 16, 16, stream=0)
    assert e.value.code == binding.HSTU_ERR_UNSUPPORTED
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_attn_bwd(16, 16, 16, 16, off, 1, 0, 64, 4, 1.0, 1.0, 16, 16, 16, stream=0)
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG
    binding.hstu_attn_bwd(0, 0, 0, 0, np.zeros(1, np.int32), 0, 2, 64, 0, 1.0, 1.0, 0, 0, 0, stream=0)


def test_bwd_rab_validation_before_any_cuda_call():
    off = np.array([0, 4], np.int32)
    good = dict(ts=16, pos=16, npos=8, time=16, ntime=8, dpos=32, dtime=32)
    bad = [dict(ts=0), dict(pos=0), dict(ts=18), dict(npos=0), dict(ntime=33), dict(dpos=0),
           dict(dtime=0), dict(dpos=34), dict(dtime=2)]
    for kw in bad:
        a = dict(good)
        a.update(kw)
        rab = binding.ctypes.pointer(binding._Rab(a["ts"], a["pos"], a["npos"], a["time"], a["ntime"]))
        code = binding.lib().hstu_attn_bwd_ex(16, 16, 16, 16, off.ctypes.data, None, 1, 2, 64, 4, rab,
                                              1.0, 1.0, 16, 16, 16, a["dpos"], a["dtime"], None)
        assert code == binding.HSTU_ERR_INVALID_ARG, kw
        code = binding.lib().hstu_attn_bwd_plan_ex(None, 16, 16, 16, 16, rab, 1.0, 1.0, 16, 16, 16,
                                                   a["dpos"], a["dtime"], None)
        assert code == binding.HSTU_ERR_INVALID_ARG, kw
    # without the bias the table gradients are not looked at
    binding.hstu_attn_bwd_ex(0, 0, 0, 0, np.zeros(1, np.int32), 0, 2, 64, 0, 1.0, 1.0, 0, 0, 0,
                             stream=0)


# ------------------------------------------------ candidates only (M-FALCON's cached history)
@pytest.mark.parametrize("seed", range(8))
def test_candidates_only_worklist_bit_exact_random(seed):
    rng = np.random.default_rng(1300 + seed)
    nb = int(rng.integers(0, 20))
    lengths = rng.integers(0, 700, size=nb)
    # edges: no candidates, all candidates, history a multiple of 128
    nt = [int(rng.choice([0, n, n % 128, rng.integers(0, n + 1)])) if n else 0 for n in lengths]
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    heads = int(rng.integers(1, 4))
    items, hist = binding.hstu_worklist_build_candidates(off, np.array(nt, np.int32), heads)
    ref_items, ref_hist = oracle_worklist.items_candidates(off, nt, heads)
    assert np.array_equal(items, ref_items.reshape(-1, 4))
    assert np.array_equal(hist, ref_hist)


def test_candidates_only_worklist_is_a_subsequence_of_the_candidate_one():
    w, nt = workloads.candidate_workload()
    full, fh = binding.hstu_worklist_build_targets(w.offsets, nt, w.heads)
    part, ph = binding.hstu_worklist_build_candidates(w.offsets, nt, w.heads)
    keys = {tuple(r) for r in full.tolist()}
    assert all(tuple(r) in keys for r in part.tolist())
    pos = [full.tolist().index(r) for r in part.tolist()[:50]]
    assert pos == sorted(pos)
    # each sequence keeps its candidates' blocks: 1024 candidates span 8 or 9 blocks
    per_seq = len(part) // w.heads
    assert 8 * w.batch <= per_seq <= 9 * w.batch


def test_candidates_only_plan_flag_validation_before_any_cuda_call():
    off = np.array([0, 300], np.int32)
    nt = np.array([20], np.int32)
    for flags, targets in ((binding.HSTU_PLAN_CANDIDATES_ONLY, None),
                           (binding.HSTU_PLAN_CANDIDATES_ONLY | binding.HSTU_PLAN_NORM_GATE, nt),
                           (binding.HSTU_PLAN_CANDIDATES_ONLY | binding.HSTU_PLAN_BACKWARD, nt),
                           (8, nt)):
        with pytest.raises(binding.HstuError) as e:
            binding.hstu_plan_create_ex(off, targets, 1, 2, 64, 300, flags)
        assert e.value.code == binding.HSTU_ERR_INVALID_ARG, flags



# ------------------------------------------------ backward with candidates
@pytest.mark.parametrize("seed", range(8))
def test_bwd_candidate_worklist_bit_exact_random(seed):
    rng = np.random.default_rng(1500 + seed)
    nb = int(rng.integers(0, 20))
    lengths = rng.integers(0, 700, size=nb)
    nt = [int(rng.choice([0, n, n % 128, rng.integers(0, n + 1)])) if n else 0 for n in lengths]
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    heads = int(rng.integers(1, 4))
    items, hist = binding.hstu_worklist_build_bwd_targets(off, np.array(nt, np.int32), heads)
    ref_items, ref_hist = oracle_worklist.items_bwd_targets(off, nt, heads)
    assert np.array_equal(items, ref_items.reshape(-1, 4))
    assert np.array_equal(hist, ref_hist)


def test_bwd_candidate_worklist_without_candidates_is_the_causal_one():
    w = workloads.workload("serving")
    items, hist = binding.hstu_worklist_build_bwd_targets(w.offsets, np.zeros(w.batch, np.int32),
                                                          w.heads)
    assert np.array_equal(items, binding.hstu_worklist_build_bwd(w.offsets, w.heads))
    assert np.array_equal(hist, items[:, 1])


def test_bwd_candidates_validation():
    off = np.array([0, 300], np.int32)
    for nt in ([-1], [301]):
        with pytest.raises(binding.HstuError) as e:
            binding.hstu_worklist_build_bwd_targets(off, np.array(nt, np.int32), 2)
        assert e.value.code == binding.HSTU_ERR_INVALID_ARG, nt


@pytest.mark.parametrize("name", workloads.WORKLOAD_NAMES)
def test_pair_worklist_bit_exact_vs_oracle(name):
    w = workloads.workload(name)
    got = binding.hstu_worklist_build_pairs(w.offsets, w.heads)
    ref = oracle_worklist.items_pairs(w.offsets, w.heads)
    assert got.dtype == np.int32 and got.shape == ref.shape
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("seed", range(12))
def test_pair_worklist_bit_exact_random(seed):
    rng = np.random.default_rng(500 + seed)
    nb = int(rng.integers(0, 40))
    lengths = rng.integers(0, 1200, size=nb) * (rng.random(nb) > 0.2)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    heads = int(rng.integers(1, 6))
    got = binding.hstu_worklist_build_pairs(off, heads)
    ref = oracle_worklist.items_pairs(off, heads)
    assert np.array_equal(got.reshape(-1, 4), ref.reshape(-1, 4))
