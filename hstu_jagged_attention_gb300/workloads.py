"""Seeded synthetic workloads for HSTU jagged causal attention.

This module only draws random numbers: sequence lengths, and Q/K/V values
rounded to bf16.  It holds none of the attention arithmetic, so both the
CUDA path and the fp64 oracle can take their inputs from it without sharing
any of the method's code.

The five workloads follow the shapes the pages measure or describe:

* ``tiny``    -- 4 sequences of lengths {7, 33, 64, 1}, 2 heads, d = 32.
* ``dense``   -- the page's QKV(16, 4, 4096, 64) shape stored as a jagged
  batch with uniform offsets (ai6s.net "HSTU fused operator" post, sections
  2.2 and 3.2).
* ``skewed``  -- 128 sequences, lengths i.i.d. from a truncated power law
  p(n) ~ n^-1.5 on [16, 8192], 4 heads, d = 128 (skewed user-history lengths,
  HSTU paper section 3.2).
* ``long``    -- 4 sequences of 10240..20480 tokens, 4 heads, d = 64 (the
  post's "0 < s <= 20480" range, section 3.1).
* ``serving`` -- 512 sequences with log-normal lengths (median 512,
  sigma 1.0) clipped to [1, 8192], 2 heads, d = 64.

Seeds: lengths use ``seed = index`` (0..4); Q, K and V use
``seed = 1000 + index`` and are drawn in that order.  Values are fp32
standard normals times sigma, rounded to bf16 with round-to-nearest-even.

One more workload exercises the candidate (M-FALCON) mask of the HSTU paper
(section 3.4, Appendix H): ``candidates`` -- 32 sequences, each a user
history of 2048..8192 tokens followed by b_m = 1024 ranking candidates
(the appendix takes b_m of the order of n), 4 heads, d = 64.  Its lengths
use seed 5 and Q, K, V seed 1005.

The layer's output stage, Norm(A V) (.) U (HSTU paper section 3), takes
three more inputs, drawn by ``draw_norm_gate`` from ``default_rng(2000 +
index)`` in this order: U of Q's shape, fp32 standard normals rounded to
bf16; gamma = 1 + 0.1 N(0, 1) and beta = 0.1 N(0, 1), fp32, heads * d each.
The layer norm's eps is NORM_EPS = 1e-6.

The relative attention bias (HSTU paper section 3, rab_{p,t}) takes
timestamps and two tables, drawn by ``draw_rab`` from
``default_rng(3000 + index)``:
- Each sequence starts at a uniform integer time in [0, 10^9) seconds.
- Its tokens follow in time order with log-normal gaps, exp(N(6, 2.5^2))
  seconds (a median of about 7 minutes), summed and capped below 2^31.
- The tables have RAB_BUCKETS = 32 entries each, 0.2 N(0, 1), fp32.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

WORKLOAD_NAMES = ("tiny", "dense", "skewed", "long", "serving")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    batch: int
    heads: int
    d: int
    sigma: float
    lengths: np.ndarray  # int64[batch]
    alpha: float
    inv_n: float

    @property
    def offsets(self) -> np.ndarray:
        off = np.zeros(self.batch + 1, dtype=np.int32)
        np.cumsum(self.lengths, out=off[1:])
        return off

    @property
    def total(self) -> int:
        return int(self.lengths.sum())

    @property
    def max_seqlen(self) -> int:
        return int(self.lengths.max()) if self.batch else 0

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "batch": self.batch,
            "heads": self.heads,
            "d": self.d,
            "total_tokens": self.total,
            "max_seqlen": self.max_seqlen,
            "alpha": self.alpha,
            "inv_n": self.inv_n,
            "sigma": self.sigma,
        }


def _lengths(name: str, rng: np.random.Generator) -> np.ndarray:
    if name == "tiny":
        return np.array([7, 33, 64, 1], dtype=np.int64)
    if name == "dense":
        return np.full(16, 4096, dtype=np.int64)
    if name == "skewed":
        support = np.arange(16, 8193, dtype=np.int64)
        pmf = support.astype(np.float64) ** -1.5
        pmf /= pmf.sum()
        return rng.choice(support, size=128, p=pmf).astype(np.int64)
    if name == "long":
        return rng.integers(10240, 20481, size=4).astype(np.int64)
    if name == "serving":
        raw = np.exp(math.log(512.0) + rng.standard_normal(512))
        return np.clip(np.rint(raw), 1, 8192).astype(np.int64)
    raise KeyError(f"unknown workload {name!r}; expected one of {WORKLOAD_NAMES}")


_SHAPES = {
    # name: (heads, d, sigma)
    "tiny": (2, 32, 1.0),
    "dense": (4, 64, 1.0),
    "skewed": (4, 128, 0.5),
    "long": (4, 64, 1.0),
    "serving": (2, 64, 1.0),
}


def workload(name: str) -> Workload:
    """The named workload's shape, lengths and scalars (no tensors drawn)."""
    index = WORKLOAD_NAMES.index(name)
    heads, d, sigma = _SHAPES[name]
    lengths = _lengths(name, np.random.default_rng(index))
    max_len = int(lengths.max())
    alpha = 1.0 / math.sqrt(d)
    if name == "tiny":
        inv_n = 1.0 / 64
    elif name == "dense":
        inv_n = 1.0 / 4096
    elif name == "serving":
        inv_n = 1.0 / 8192
    else:  # skewed, long: 1 / (largest sampled length)
        inv_n = 1.0 / max_len
    return Workload(name, index, len(lengths), heads, d, sigma, lengths, alpha, inv_n)


def custom(lengths, heads: int, d: int, sigma: float = 1.0, alpha: float | None = None,
           inv_n: float | None = None, name: str = "custom") -> Workload:
    """A workload with caller-chosen lengths (tests: ragged tails, empties)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    max_len = int(lengths.max()) if len(lengths) else 1
    return Workload(name, -1, len(lengths), heads, d, sigma, lengths,
                    1.0 / math.sqrt(d) if alpha is None else float(alpha),
                    1.0 / max(max_len, 1) if inv_n is None else float(inv_n))


def bf16_round(x: np.ndarray):
    """fp32 array -> torch bf16 tensor (round to nearest even)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def draw_qkv(w: Workload, seed: int | None = None):
    """Q, K, V as CPU torch bf16 tensors of shape (total, heads, d).

    Drawn from ``default_rng(1000 + index)`` (or ``seed``) in the order Q, K, V.
    """
    rng = np.random.default_rng(1000 + w.index if seed is None else seed)
    shape = (w.total, w.heads, w.d)
    out = []
    for _ in range(3):
        x = rng.standard_normal(shape, dtype=np.float32)
        if w.sigma != 1.0:
            x *= np.float32(w.sigma)
        out.append(bf16_round(x))
    return tuple(out)


CANDIDATES_INDEX = 5
CANDIDATES_BM = 1024


def candidate_workload() -> tuple[Workload, np.ndarray]:
    """The ``candidates`` workload and its int32 num_targets (see the module doc)."""
    rng = np.random.default_rng(CANDIDATES_INDEX)
    hist = rng.integers(2048, 8193, size=32).astype(np.int64)
    lengths = hist + CANDIDATES_BM
    w = Workload("candidates", CANDIDATES_INDEX, len(lengths), 4, 64, 1.0, lengths,
                 1.0 / math.sqrt(64), 1.0 / int(lengths.max()))
    return w, np.full(len(lengths), CANDIDATES_BM, dtype=np.int32)


NORM_EPS = 1e-6


def draw_norm_gate(w: Workload, seed: int | None = None):
    """U (CPU torch bf16, (total, heads, d)), gamma and beta (fp32 numpy,
    heads * d) for the output stage; ``default_rng(2000 + index)`` or ``seed``."""
    rng = np.random.default_rng(2000 + w.index if seed is None else seed)
    u = bf16_round(rng.standard_normal((w.total, w.heads, w.d), dtype=np.float32))
    width = w.heads * w.d
    gamma = (1.0 + 0.1 * rng.standard_normal(width)).astype(np.float32)
    beta = (0.1 * rng.standard_normal(width)).astype(np.float32)
    return u, gamma, beta


RAB_BUCKETS = 32


def draw_rab(w: Workload, seed: int | None = None, backwards: float = 0.0):
    """Timestamps (int32 numpy, one per token) and the position and time
    tables (fp32 numpy, RAB_BUCKETS each); ``default_rng(3000 + index)`` or
    ``seed``.  ``backwards``: the fraction of gaps drawn negative (tests of
    the clamp at dt = 0)."""
    rng = np.random.default_rng(3000 + w.index if seed is None else seed)
    ts = np.zeros(w.total, dtype=np.int64)
    off = w.offsets.astype(np.int64)
    for b in range(w.batch):
        n = int(w.lengths[b])
        start = int(rng.integers(0, 10 ** 9))
        gaps = np.exp(rng.normal(6.0, 2.5, size=n)).astype(np.int64)
        if backwards:
            gaps[rng.random(n) < backwards] *= -1
        ts[off[b]:off[b + 1]] = np.clip(start + np.cumsum(gaps), 0, 2 ** 31 - 1)
    pos = (0.2 * rng.standard_normal(RAB_BUCKETS)).astype(np.float32)
    time = (0.2 * rng.standard_normal(RAB_BUCKETS)).astype(np.float32)
    return ts.astype(np.int32), pos, time
