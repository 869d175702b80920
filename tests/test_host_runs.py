"""CPU: the runs of whole sequences the host-buffer forward takes.

hstu_attn_fwd_host splits the sequences into runs with about equal token
counts, so that each run's copies overlap another run's kernel; the GPU
tests check that the output does not depend on the split.  These tests pin
the split itself (hstu_host_runs, no CUDA call): hand-worked cases, the
rule the header states, and its balance bound.
"""
import numpy as np
import pytest

from hstu_jagged_attention_gb300 import binding


def offsets_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def test_hand_worked_runs():
    # 3008 tokens in 3 runs: thresholds 1002 and 2005; sequence 2 is the
    # first to start past either, so run 1 is empty
    assert binding.hstu_host_runs(offsets_of([5, 3000, 1, 2]), 3).tolist() == [0, 2, 2, 4]
    # 800 tokens of equal sequences in 4 runs: thresholds 200, 400, 600
    assert binding.hstu_host_runs(offsets_of([100] * 8), 4).tolist() == [0, 2, 4, 6, 8]
    # 0 asks for the default, min(batch, 4)
    assert binding.hstu_host_runs(offsets_of([100] * 8), 0).tolist() == [0, 2, 4, 6, 8]
    # more runs than sequences: capped at 3 runs; 16 tokens, thresholds 5
    # and 10: sequence 1 (empty, at token 7) opens run 1, and no sequence
    # starts at or past 10, so run 1 takes the rest and run 2 is empty
    assert binding.hstu_host_runs(offsets_of([7, 0, 9]), 10).tolist() == [0, 1, 3, 3]
    assert binding.hstu_host_runs(offsets_of([7, 0, 9]), 0).tolist() == [0, 1, 3, 3]
    # one run: everything
    assert binding.hstu_host_runs(offsets_of([7, 0, 9]), 1).tolist() == [0, 3]
    # no sequences
    assert binding.hstu_host_runs(offsets_of([]), 0).tolist() == [0]


@pytest.mark.parametrize("seed", range(20))
def test_random_runs_follow_the_rule_and_balance(seed):
    rng = np.random.default_rng(1300 + seed)
    lengths = rng.integers(0, 5000, size=int(rng.integers(1, 300)))
    lengths[rng.random(len(lengths)) < 0.1] = 0
    off = offsets_of(lengths)
    batch, total = len(lengths), int(off[-1])
    n_chunks = int(rng.integers(0, 12))
    first = binding.hstu_host_runs(off, n_chunks)
    n = min(batch, n_chunks if n_chunks > 0 else 4)
    assert len(first) == n + 1 and first[0] == 0 and first[-1] == batch
    assert np.all(np.diff(first) >= 0)
    for c in range(1, n):
        # the first sequence at or past the threshold, or the previous
        # run's end if that is later
        thr = total * c // n
        b = int(np.searchsorted(off[:batch], thr, side="left"))
        assert first[c] == max(b, first[c - 1]), (c, thr)
    run_tokens = off[first[1:]] - off[first[:-1]]
    assert run_tokens.sum() == total
    assert run_tokens.max(initial=0) <= total / n + lengths.max(initial=0) + 1


def test_errors():
    with pytest.raises(binding.HstuError):
        binding.hstu_host_runs(offsets_of([5, 6]), -1)
    with pytest.raises(binding.HstuError):
        binding.hstu_host_runs(np.array([1, 5], dtype=np.int32), 0)  # not starting at 0
    with pytest.raises(binding.HstuError):
        binding.hstu_host_runs(np.array([0, 9, 5], dtype=np.int32), 0)  # decreasing
