"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance per element: |gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref) (see
tests/parity.py).  Small cases and the full-size workloads are compared
element by element over the whole output; the full-size workloads are also
compared on a uniform random sample of rows plus edge rows (the sampled
oracle), in the launch configuration the benchmark times (a prebuilt plan
over device buffers).
"""
import numpy as np
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


def _draw(w, seed=None):
    q, k, v = workloads.draw_qkv(w, seed)
    return (q, k, v), parity.to_device(q, k, v)


def test_tiny_workload_full():
    w = workloads.workload("tiny")
    (q, k, v), (qd, kd, vd) = _draw(w)
    out = parity.run_plan(w, qd, kd, vd)
    parity.full_check(w, q, k, v, out)
    parity.assert_device_ok()


RAGGED = [1, 127, 128, 129, 300, 0, 513, 700, 2, 256, 255]


@pytest.mark.parametrize("d", [32, 64, 128])
def test_ragged_multi_tile_full(d):
    w = workloads.custom(RAGGED, heads=3, d=d, sigma=1.0 if d < 128 else 0.5)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=50 + d)
    out = parity.run_plan(w, qd, kd, vd)
    parity.full_check(w, q, k, v, out)
    parity.assert_device_ok()


@pytest.mark.parametrize("d", [32, 64, 128])
def test_many_short_sequences_full(d):
    rng = np.random.default_rng(d)
    lengths = rng.integers(0, 200, size=300)
    lengths[::7] = 1
    lengths[::11] = 0
    w = workloads.custom(lengths, heads=2, d=d)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=70 + d)
    out = parity.run_plan(w, qd, kd, vd)
    parity.full_check(w, q, k, v, out)


@pytest.mark.parametrize("name", ["dense", "skewed", "long", "serving"])
def test_full_size_workloads_every_element(name):
    # Every output element of the full-size workload against the threaded
    # fp64 oracle (tens of seconds on the host cores), in the launch
    # configuration the benchmark times.
    w = workloads.workload(name)
    (q, k, v), (qd, kd, vd) = _draw(w)
    out = parity.run_plan(w, qd, kd, vd)
    parity.assert_device_ok()
    worst = parity.full_check(w, q, k, v, out)
    print(f"\n{name}: worst err/tol over every element {worst:.3f}")


@pytest.mark.parametrize("name", ["dense", "skewed", "long", "serving"])
def test_full_size_workloads_sampled(name):
    w = workloads.workload(name)
    (q, k, v), (qd, kd, vd) = _draw(w)
    out = parity.run_plan(w, qd, kd, vd)
    parity.assert_device_ok()
    parity.sampled_check(w, q, k, v, out, n_random=256, seed=1)


def test_call_path_equals_plan_path_and_device_offsets():
    w = workloads.custom(RAGGED, heads=2, d=64)
    _, (qd, kd, vd) = _draw(w, seed=3)
    a = parity.run_plan(w, qd, kd, vd)
    b = parity.run_call(w, qd, kd, vd)
    c = parity.run_call(w, qd, kd, vd, offsets=torch.as_tensor(w.offsets, device="cuda"))
    assert torch.equal(a, b) and torch.equal(a, c)


def test_deterministic():
    w = workloads.custom(RAGGED, heads=2, d=128, sigma=0.5)
    _, (qd, kd, vd) = _draw(w, seed=4)
    a = parity.run_plan(w, qd, kd, vd)
    b = parity.run_plan(w, qd, kd, vd)
    assert torch.equal(a, b)


def test_alpha_zero_gives_exact_zero():
    w = workloads.custom(RAGGED, heads=2, d=64, alpha=0.0)
    _, (qd, kd, vd) = _draw(w, seed=5)
    out = parity.run_plan(w, qd, kd, vd)
    assert torch.count_nonzero(out.float()) == 0


def test_causality_bit_exact():
    # Rows <= i of a sequence ignore keys and values after i (the triangular
    # diagonal block is a select, and P = 0 times finite V is an exact zero).
    w = workloads.custom([700, 300], heads=2, d=64)
    _, (qd, kd, vd) = _draw(w, seed=6)
    base = parity.run_plan(w, qd, kd, vd)
    for i in (0, 127, 128, 450, 698):
        k2, v2 = kd.clone(), vd.clone()
        k2[i + 1:700] = torch.randn_like(k2[i + 1:700].float()).to(k2.dtype) * 3
        v2[i + 1:700] = torch.randn_like(v2[i + 1:700].float()).to(v2.dtype) * 3
        out = parity.run_plan(w, qd, k2, v2)
        assert torch.equal(out[: i + 1], base[: i + 1]), i
        assert torch.equal(out[700:], base[700:])


def test_nonfinite_values_in_next_sequence_do_not_leak():
    # The last key block of a sequence extends into the next sequence's rows;
    # their K and V must never reach this sequence's output, even when they
    # are Inf or NaN.
    w = workloads.custom([200, 100], heads=2, d=64)
    _, (qd, kd, vd) = _draw(w, seed=7)
    base = parity.run_plan(w, qd, kd, vd)
    k2, v2 = kd.clone(), vd.clone()
    k2[200:] = float("inf")
    v2[200:] = float("nan")
    out = parity.run_plan(w, qd, k2, v2)
    assert torch.equal(out[:200], base[:200])


def test_empty_and_single_token_sequences():
    w = workloads.custom([0, 1, 0, 0, 1, 1, 0, 3, 0], heads=4, d=32, inv_n=0.5)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=8)
    out = parity.run_plan(w, qd, kd, vd)
    parity.full_check(w, q, k, v, out)
    out2 = parity.run_call(w, qd, kd, vd)
    assert torch.equal(out, out2)


def test_all_empty_and_zero_batch_are_noops():
    w = workloads.custom([0, 0, 0], heads=2, d=64)
    z = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    parity.run_plan(w, z, z, z, out=z)
    parity.run_call(w, z, z, z)
    binding.hstu_attn_fwd(0, 0, 0, np.zeros(1, np.int32), 0, 2, 64, 0, 1.0, 1.0, 0)


def test_only_valid_rows_written():
    # out has 64 canary rows after the last token; every valid row must be
    # overwritten and no canary byte touched.
    w = workloads.custom([130, 1, 257], heads=2, d=128, sigma=0.5)
    _, (qd, kd, vd) = _draw(w, seed=9)
    canary = torch.full((w.total + 64, 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    canary_bits = canary.view(torch.int16).clone()
    out = canary[: w.total]
    parity.run_plan(w, qd, kd, vd, out=out)
    assert torch.isfinite(out.float()).all()
    assert torch.equal(canary.view(torch.int16)[w.total:], canary_bits[w.total:])


def test_head_major_dense_input_via_permute():
    # A dense (b, heads, s, d) head-major tensor is the uniform-offsets case
    # once permuted to token-major (b*s, heads, d).
    b, H, s, d = 2, 3, 200, 64
    w = workloads.custom([s] * b, heads=H, d=d)
    g = torch.Generator().manual_seed(10)
    Qh, Kh, Vh = (torch.randn((b, H, s, d), generator=g).to(torch.bfloat16) for _ in range(3))
    tok = lambda x: x.permute(0, 2, 1, 3).reshape(b * s, H, d).contiguous()
    q, k, v = tok(Qh), tok(Kh), tok(Vh)
    out = parity.run_plan(w, *parity.to_device(q, k, v))
    parity.full_check(w, q, k, v, out)


def test_max_length_sequence_sampled():
    # the longest sequence the page's range allows (s = 20480), 1 head
    w = workloads.custom([20480], heads=1, d=64, inv_n=1 / 20480)
    (q, k, v), (qd, kd, vd) = _draw(w, seed=11)
    out = parity.run_plan(w, qd, kd, vd)
    parity.sampled_check(w, q, k, v, out, n_random=128, seed=2)
