"""hstu_attn_fwd_noalloc: the forward for callers that cannot allocate.

Some callers own all device memory themselves (a serving process with a
fixed memory budget, or a framework whose allocator must not be bypassed)
and cannot let the library call cudaMalloc or cudaMallocAsync.  This entry
point keeps the work list in a fixed array inside the library instead.
Its output must match hstu_attn_fwd's, call after call, within the parity
tolerance the other GPU tests use, and the fp64 oracle's element by
element.  This file is collected last so that a failure here does not hide
the results of the other tests.
"""
import numpy as np
import pytest
import torch

from hstu_jagged_attention_gb300 import binding, build, workloads
from tests import parity

pytestmark = pytest.mark.gpu


def _existing(w, q, k, v):
    out = torch.empty_like(q)
    binding.hstu_attn_fwd(q, k, v, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha, w.inv_n, out)
    return out


def _noalloc(w, q, k, v):
    out = torch.empty_like(q)
    binding.hstu_attn_fwd_noalloc(q, k, v, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                  w.inv_n, out)
    return out


def _assert_close(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(r ** 2)))
    assert np.isfinite(g).all()
    assert parity.ratio(g, r, rms).max() <= 1.0


def test_noalloc_matches_existing_entry_on_two_calls_in_a_row():
    build.build()
    # the first call covers more work items than the second, so a stale tail
    # left in the shared array by call 1 must not leak into call 2
    first = workloads.custom([1, 127, 128, 129, 300, 0, 513, 700, 2], heads=3, d=64)
    second = workloads.custom([40, 0, 260, 5], heads=2, d=128, sigma=0.5)
    for w, seed in ((first, 31), (second, 32)):
        q, k, v = parity.to_device(*workloads.draw_qkv(w, seed=seed))
        got = _noalloc(w, q, k, v)
        ref = _existing(w, q, k, v)
        torch.cuda.synchronize()
        _assert_close(got, ref)
        parity.full_check(w, q, k, v, got)
    assert binding.hstu_last_status() == (binding.HSTU_OK, 0)


def test_noalloc_rejects_work_lists_beyond_capacity_and_device_offsets():
    build.build()
    # 513 sequences x 128 heads x 1 block = 65,664 items > 65,536
    w = workloads.custom([1] * 513, heads=128, d=32)
    q = torch.zeros((w.total, w.heads, w.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_attn_fwd_noalloc(q, q, q, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, 1.0,
                                      1.0, torch.empty_like(q))
    assert e.value.code == binding.HSTU_ERR_CAPACITY
    off_dev = torch.as_tensor(w.offsets, device="cuda")
    with pytest.raises(binding.HstuError) as e:
        binding.hstu_attn_fwd_noalloc(q, q, q, off_dev.data_ptr(), w.batch, w.heads, w.d,
                                      w.max_seqlen, 1.0, 1.0, torch.empty_like(q))
    assert e.value.code == binding.HSTU_ERR_INVALID_ARG
