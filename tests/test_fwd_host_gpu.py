"""GPU: the forward from host buffers to host buffers (hstu_attn_fwd_host).

The call splits the sequences into runs of whole sequences, copies each
run's q, k, v rows in on internal streams, runs the forward on the
caller's stream and copies the out rows back on another.  Every output row
comes from the same kernel arithmetic as hstu_attn_fwd, so the two must
agree bit for bit, whatever the number of runs; one case is also checked
element by element against the fp64 oracle.
"""
import pytest
import torch

from hstu_jagged_attention_gb300 import binding, build, workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.hstu_set_wait_timeout_ns(0)
    yield
    parity.assert_device_ok()


RAGGED = [300, 0, 513, 1, 256, 700, 90, 129, 0, 640, 385, 2]


def _host(t, pinned=True):
    t = t.contiguous()
    return t.pin_memory() if pinned else t.clone()


def _run_host(w, q, k, v, n_chunks, pinned=True, out_fill=float("nan")):
    qh, kh, vh = (_host(t, pinned) for t in (q, k, v))
    out_h = _host(torch.full(q.shape, out_fill, dtype=q.dtype), pinned)
    qd, kd, vd, od = (torch.empty(q.shape, dtype=q.dtype, device="cuda") for _ in range(4))
    binding.hstu_attn_fwd_host(qh, kh, vh, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                               w.inv_n, out_h, qd, kd, vd, od, n_chunks=n_chunks)
    torch.cuda.synchronize()
    parity.assert_device_ok()
    return out_h


def _run_device(w, q, k, v):
    return parity.run_call(w, *parity.to_device(q, k, v)).cpu()


@pytest.mark.parametrize("d", [32, 64, 128])
def test_host_call_equals_device_call_for_any_chunking(d):
    w = workloads.custom(RAGGED, heads=2, d=d)
    q, k, v = workloads.draw_qkv(w, seed=1200 + d)
    ref = _run_device(w, q, k, v)
    for n_chunks in (0, 1, 2, 3, 5, len(RAGGED), 100):
        got = _run_host(w, q, k, v, n_chunks)
        assert torch.equal(got, ref), n_chunks


def test_host_call_against_the_oracle_every_element():
    w = workloads.custom(RAGGED, heads=2, d=64)
    q, k, v = workloads.draw_qkv(w, seed=1210)
    got = _run_host(w, q, k, v, 3)
    parity.full_check(w, q, k, v, got)


def test_pageable_host_buffers():
    w = workloads.custom([129, 900, 31], heads=2, d=64)
    q, k, v = workloads.draw_qkv(w, seed=1220)
    assert torch.equal(_run_host(w, q, k, v, 2, pinned=False), _run_device(w, q, k, v))


def test_one_sequence_holding_most_tokens_leaves_runs_empty():
    # runs split by token count: with one long sequence some runs hold none
    w = workloads.custom([5, 3000, 1, 2], heads=2, d=64)
    q, k, v = workloads.draw_qkv(w, seed=1230)
    ref = _run_device(w, q, k, v)
    for n_chunks in (2, 3, 4):
        assert torch.equal(_run_host(w, q, k, v, n_chunks), ref), n_chunks


def test_two_calls_in_a_row_on_one_stream():
    w = workloads.custom(RAGGED, heads=2, d=64)
    qa, ka, va = workloads.draw_qkv(w, seed=1240)
    qb, kb, vb = workloads.draw_qkv(w, seed=1241)
    hosts = [[_host(t) for t in trio] for trio in ((qa, ka, va), (qb, kb, vb))]
    outs = [_host(torch.empty_like(qa)) for _ in range(2)]
    dev = [torch.empty(qa.shape, dtype=qa.dtype, device="cuda") for _ in range(4)]
    for (qh, kh, vh), oh in zip(hosts, outs):
        binding.hstu_attn_fwd_host(qh, kh, vh, w.offsets, w.batch, w.heads, w.d, w.max_seqlen,
                                   w.alpha, w.inv_n, oh, *dev, n_chunks=3)
    torch.cuda.synchronize()
    parity.assert_device_ok()
    assert torch.equal(outs[0], _run_device(w, qa, ka, va))
    assert torch.equal(outs[1], _run_device(w, qb, kb, vb))


def test_empty_batch_and_argument_errors():
    w = workloads.custom([0, 0], heads=2, d=64)
    z = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
    zd = torch.zeros(8, 2, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(z, 3.0)
    binding.hstu_attn_fwd_host(z, z, z, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                               w.inv_n, out, zd, zd, zd, zd)
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    w = workloads.custom([3, 5], heads=2, d=64)
    with pytest.raises(binding.HstuError):
        binding.hstu_attn_fwd_host(z, z, z, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                   w.inv_n, out, zd, zd, zd, zd, n_chunks=-1)
    lib = binding.lib()
    dev_off = torch.as_tensor(w.offsets, device="cuda")
    rc = lib.hstu_attn_fwd_host(z.data_ptr(), z.data_ptr(), z.data_ptr(), dev_off.data_ptr(), w.batch,
                                w.heads, w.d, w.max_seqlen, w.alpha, w.inv_n, out.data_ptr(),
                                zd.data_ptr(), zd.data_ptr(), zd.data_ptr(), zd.data_ptr(), 0, None)
    assert rc == binding.HSTU_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        binding.hstu_attn_fwd_host(zd, z, z, w.offsets, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                   w.inv_n, out, zd, zd, zd, zd)


def test_full_size_dense_equals_device_call():
    # the configuration the benchmark's end-to-end leg times
    w = workloads.workload("dense")
    q, k, v = workloads.draw_qkv(w)
    assert torch.equal(_run_host(w, q, k, v, 0), _run_device(w, q, k, v))
