"""The benchmark's work counts against brute-force counts of kept pairs.

causal_flops: 4 d FLOP per kept (query, key) pair and head (HSTU paper
section 3.1 and the post's FLOP convention: two matmuls of 2 d each);
bwd_flops: 10 d (the recomputed S and dP, then dV, dK and dQ);
candidate_row_flops: 4 d over the candidates' rows only.  The kept pairs
are those of the causal mask, or of the candidate mask (HSTU paper
Appendix H): j <= i and (j < hist or j == i).
"""
import numpy as np
import pytest

import bench
from hstu_jagged_attention_gb300 import workloads


def _kept(n, hist):
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return (j <= i) & ((j < hist) | (j == i))


@pytest.mark.parametrize("seed", range(6))
def test_flop_counts_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(0, 300, size=int(rng.integers(1, 8)))
    heads, d = int(rng.integers(1, 5)), int(rng.choice([32, 64, 128]))
    w = workloads.custom(lengths, heads=heads, d=d)
    nt = np.array([int(rng.integers(0, n + 1)) for n in lengths], dtype=np.int32)
    causal = sum(int(_kept(n, n).sum()) for n in lengths)
    masked = sum(int(_kept(n, n - t).sum()) for n, t in zip(lengths, nt))
    cand_rows = sum(int(_kept(n, n - t)[n - t:].sum()) for n, t in zip(lengths, nt))
    assert bench.causal_flops(w) == pytest.approx(4 * d * heads * causal)
    assert bench.causal_flops(w, nt) == pytest.approx(4 * d * heads * masked)
    assert bench.bwd_flops(w) == pytest.approx(10 * d * heads * causal)
    assert bench.bwd_flops(w, nt) == pytest.approx(10 * d * heads * masked)
    assert bench.candidate_row_flops(w, nt) == pytest.approx(4 * d * heads * cand_rows)


def test_dense_workload_counts():
    w = workloads.workload("dense")
    # 16 sequences of 4096 tokens, 4 heads, d = 64: 137.47 causal GFLOP
    assert bench.causal_flops(w) / 1e9 == pytest.approx(137.47, rel=1e-4)
    assert bench.algorithmic_bytes(w) == 8 * 64 * 4 * 65536


def test_roofline_entry_picks_the_bound_by_intensity():
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}   # ridge 250 FLOP/B
    hi = bench.roofline_entry(flops=1e12, nbytes=1e9, ms=1.0, peaks=peaks)   # 1000 FLOP/B
    lo = bench.roofline_entry(flops=1e10, nbytes=1e9, ms=1.0, peaks=peaks)   # 10 FLOP/B
    assert hi["bound"] == "tensor" and lo["bound"] == "hbm"
    assert hi["ridge_flop_per_byte"] == pytest.approx(250.0)
    assert hi["causal_tflops"] == pytest.approx(1000.0) and hi["pct_of_bf16_peak"] == pytest.approx(50.0)
    assert lo["hbm_gbs"] == pytest.approx(1000.0) and lo["pct_of_hbm_peak"] == pytest.approx(12.5)


def test_tiny_is_hbm_side_and_dense_tensor_side_of_the_measured_ridge():
    peaks = {"bf16_tflops": 1923.8, "hbm_gbs": 6796.9}
    for name, want in (("tiny", "hbm"), ("dense", "tensor"), ("long", "tensor")):
        w = workloads.workload(name)
        e = bench.roofline_entry(bench.causal_flops(w), bench.algorithmic_bytes(w), 1.0, peaks)
        assert e["bound"] == want, name


def test_single_thread_oracle_report_runs_bounded():
    rep = bench.cpu_single_thread_report(0.3)
    assert rep["tiny"]["cores"] == 1 and rep["dense"]["cores"] == 1
    assert rep["tiny"]["causal_tflops"] > 0 and rep["dense"]["causal_tflops"] > 0
