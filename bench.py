"""Benchmark: HSTU jagged causal attention forward on GB300.

One step = one forward over the whole workload (every (sequence, head,
query block) item; all hot-path stages run inside the one kernel).  The
default workload is the page's dense shape QKV(16, 4, 4096, 64) stored as a
jagged batch with uniform offsets.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--sweep]

Timing: W untimed warm-up steps, then K steps; each step's kernel is
bracketed by CUDA events on the launching stream and an L2 flush (a 256 MiB
write) runs between steps outside the events.  The metric is causal
TFLOP/s = 4 d heads sum_b n_b (n_b + 1) / 2 / time.  Under torchrun each
rank runs the same workload on its own GPU (weak scaling, no data-path
collective); rank 0 prints one JSON line with the max time over ranks.

The default run (the dense workload, plain forward, one GPU) also times
the five workloads the same way, one after another outside the timed
region, and reports each under ``per_config``: ms/call, causal TFLOP/s and
% of the bf16 peak, algorithmic GB/s (Q, K, V read and O written once) and
% of the copy bandwidth, and the bound its arithmetic intensity selects
against the ridge of the measured peaks.  ``cpu_baseline_single_thread``
times the oracle on one host thread (tiny whole, dense sampled).

``--impl reference`` times the fp64 CPU oracle (the only reference this
method has) on the host cores, each step a bounded sample of rows of the
same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hstu_jagged_attention_gb300 import workloads  # noqa: E402

METRIC = "HSTU jagged causal attn fwd: TFLOPS & % GB300 BF16 tensor peak; ms/call"
UNIT = "TFLOP/s"
KERNEL_SOURCE = os.path.join(ROOT, "hstu_jagged_attention_gb300", "csrc", "hstu_fwd.cu")

# DRAM traffic (read + write bytes) of one launch of the forward kernel on
# the dense 16x4x4096x64 workload (plain, and the output-stage variant's
# attention kernel), from ncu captures, with the sha256 of the kernel source
# they were taken on.  The figures are reported only while the source is
# unchanged.
MEASURED_TRAFFIC = {"dense": 165165824.0, "dense+norm_gate": 195308288.0,
                    "sha256": "c2631399898c7d2194f3ac7578a141bf5a497f904784927fe09decdf98bb7afc"}


def causal_flops(w: workloads.Workload, num_targets=None) -> float:
    """4 d FLOPs per kept (query, key) pair, every head.  With candidates
    (M-FALCON mask) a sequence keeps hist (hist + 1) / 2 history pairs and,
    per candidate, hist + 1 pairs (the history and itself)."""
    L = w.lengths.astype(np.float64)
    if num_targets is None:
        pairs = np.sum(L * (L + 1) / 2.0)
    else:
        bm = np.asarray(num_targets, dtype=np.float64)
        hist = L - bm
        pairs = np.sum(hist * (hist + 1) / 2.0 + bm * (hist + 1))
    return float(4.0 * w.d * w.heads * pairs)


def candidate_row_flops(w: workloads.Workload, num_targets) -> float:
    """4 d FLOPs per kept pair of the candidates' rows only: a candidate of
    sequence b sees its hist_b history keys and itself."""
    L = w.lengths.astype(np.float64)
    bm = np.asarray(num_targets, dtype=np.float64)
    return float(4.0 * w.d * w.heads * np.sum(bm * (L - bm + 1)))


BWD_METRIC = "HSTU jagged causal attn bwd (dQ, dK, dV): TFLOPS at 10 d FLOP per kept pair; ms/call"


def bwd_flops(w: workloads.Workload, num_targets=None) -> float:
    """The backward's products per kept pair and head: S = Q K^T and dP = dO V^T
    (recomputed), dV += P^T dO, dK += dS^T Q, dQ += dS K: 5 x 2 d FLOP (the
    kept pairs of the candidate mask with ``num_targets``)."""
    return 2.5 * causal_flops(w, num_targets)


def cpu_oracle_bwd_sample(w, q, k, v, do, target_s: float, threads: int | None = None, rab=None,
                          num_targets=None):
    """The oracle's backward on the first sequences of the workload, as many
    as fit about target_s seconds (calibrated on the first one).  With the
    bias ``rab`` = (timestamps, pos, time), the tables' gradients too."""
    from oracle import reference
    threads = threads or reference.default_threads()
    off = w.offsets.astype(np.int64)

    def run(nb):
        e = int(off[nb])
        r = None if rab is None else (rab[0][:e], rab[1], rab[2])
        nt = None if num_targets is None else np.asarray(num_targets)[:nb]
        t0 = time.perf_counter()
        reference.hstu_bwd(q[:e], k[:e], v[:e], do[:e], off[:nb + 1], w.alpha, w.inv_n, threads=threads,
                           rab=r, table_grads=r is not None, num_targets=nt)
        return time.perf_counter() - t0

    nb = 1
    dt = run(nb)
    while nb < w.batch and dt * (nb + 1) / nb < target_s:
        nb = min(w.batch, max(nb + 1, int(nb * target_s / max(dt, 1e-3))))
        dt = run(nb)
    sub = workloads.custom(w.lengths[:nb], w.heads, w.d, alpha=w.alpha, inv_n=w.inv_n)
    sub_nt = None if num_targets is None else np.asarray(num_targets)[:nb]
    fl = bwd_flops(sub, sub_nt)
    desc = (f"the first {nb} of {w.batch} sequences of the {w.name} workload "
            f"({fl / 1e9:.2f} backward GFLOP), fp64 C oracle, {threads} threads")
    return fl / dt / 1e12, desc, threads, dt


def workload_by_name(name: str):
    """(workload, num_targets or None)."""
    if name == "candidates":
        return workloads.candidate_workload()
    return workloads.workload(name), None


def algorithmic_bytes(w: workloads.Workload, norm_gate: bool = False) -> float:
    # read Q, K, V (and U with the output stage) once and write O once, bf16
    return float((10.0 if norm_gate else 8.0) * w.d * w.heads * w.total)


def roofline_entry(flops: float, nbytes: float, ms: float, peaks: dict) -> dict:
    """Both roofs for one launch: causal TFLOP/s against the bf16 peak and
    algorithmic GB/s against the copy bandwidth.  The bound is the roof the
    launch's arithmetic intensity (causal FLOP per algorithmic byte) puts
    first: below the ridge peak_flops / peak_bytes it is HBM."""
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    intensity = flops / nbytes if nbytes else float("inf")
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return {"ms": ms, "causal_tflops": tflops, "pct_of_bf16_peak": 100.0 * tflops / peaks["bf16_tflops"],
            "algorithmic_bytes": nbytes, "hbm_gbs": gbs, "pct_of_hbm_peak": 100.0 * gbs / peaks["hbm_gbs"],
            "flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
            "bound": "tensor" if intensity >= ridge else "hbm"}


def time_forward_plan(w: workloads.Workload, dev, stream, flush, steps: int, warmup: int):
    """Kernel-only times (ms, one per step) of the plain forward on workload
    w, as the headline is timed: a prebuilt plan over device buffers, L2
    flushed between steps outside the events.  Returns (times, work items)."""
    import torch
    from hstu_jagged_attention_gb300 import binding
    q, k, v = (t.to(dev) for t in workloads.draw_qkv(w))
    out = torch.empty_like(q)
    plan = binding.hstu_plan_create(w.offsets, w.batch, w.heads, w.d, w.max_seqlen)
    try:
        for _ in range(warmup):
            binding.hstu_attn_fwd_plan(plan, q, k, v, w.alpha, w.inv_n, out, stream)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            binding.hstu_attn_fwd_plan(plan, q, k, v, w.alpha, w.inv_n, out, stream)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        n_items = binding.hstu_plan_num_items(plan)
    finally:
        binding.hstu_plan_destroy(plan)
    st, site = binding.hstu_last_status()
    if st != binding.HSTU_OK:
        raise RuntimeError(f"device wait gave up on the {w.name} workload (site {site})")
    return [a.elapsed_time(b) for a, b in ev], n_items


def per_config_report(dev, stream, flush, steps: int, warmup: int, peaks: dict, clock_sampler=None):
    """One entry per workload of the five configs: median ms/call, causal
    TFLOP/s, % of the bf16 peak, algorithmic GB/s, % of the copy bandwidth,
    and the bound its intensity selects."""
    rep = {}
    for name in workloads.WORKLOAD_NAMES:
        w = workloads.workload(name)
        times, n_items = time_forward_plan(w, dev, stream, flush, steps, warmup)
        ms = statistics.median(times)
        e = roofline_entry(causal_flops(w), algorithmic_bytes(w), ms, peaks)
        e.update({"ms_mean": statistics.mean(times), "ms_min": min(times), "steps": steps,
                  "work_items": n_items, "shape": w.describe()})
        rep[name] = e
    return rep


def cpu_single_thread_report(seconds: float) -> dict:
    """The oracle on one host thread (the CPU baseline plan's single-thread
    leg): the whole tiny workload, and a bounded sample of rows of dense."""
    from oracle import reference
    rep = {}
    w = workloads.workload("tiny")
    q, k, v = (t.float().numpy() for t in workloads.draw_qkv(w))
    reps, t0 = 0, time.perf_counter()
    while True:
        reference.hstu_fwd(q, k, v, w.offsets, w.alpha, w.inv_n, threads=1)
        reps += 1
        if time.perf_counter() - t0 > 0.5:
            break
    dt = (time.perf_counter() - t0) / reps
    rep["tiny"] = {"ms_per_call": dt * 1e3, "causal_tflops": causal_flops(w) / dt / 1e12, "cores": 1,
                   "sample": f"the whole tiny workload, {reps} calls, fp64 C oracle, 1 thread"}
    w = workloads.workload("dense")
    q, k, v = (t.float().numpy() for t in workloads.draw_qkv(w))
    val, desc, threads, dt = cpu_oracle_sample(w, q, k, v, seconds, seed=7, threads=1)
    rep["dense"] = {"causal_tflops": val, "cores": threads, "sample": desc,
                    "ms_per_call_extrapolated": causal_flops(w) / (val * 1e12) * 1e3}
    return rep


def kernel_sha() -> str:
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p.get("bf16_tflops_sustained"),
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, one line every 50 ms, each stamped
    with the host time it arrived; summarised over a chosen time window."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        import threading
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.perf_counter(), line.strip()))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self, t0: float, t1: float, t_warm: float) -> dict | None:
        """Summary over samples in [t0, t1] (the timed region); if fewer than
        three fall there, over [t_warm, t1] (warm-up + timed, GPU busy)."""
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = [(t, r.split(",")) for t, r in self.lines if r.count(",") >= 8]
        window = "timed region"
        sel = [r for t, r in rows if t0 - 0.05 <= t <= t1 + 0.05]
        if len(sel) < 3:
            sel = [r for t, r in rows if t_warm - 0.05 <= t <= t1 + 0.05]
            window = "warm-up + timed region"
        if not sel:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in sel) if v is not None]
        mx = [v for v in (num(r[2]) for r in sel) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i in range(4)
                          if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sel), "window": window}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(flops_per_rank: float, ms_local: float, world: int, device=None):
    """Whole-job throughput under weak scaling: every rank does flops_per_rank
    in its own time; the job takes the slowest rank's time.
    Returns (TFLOP/s over all ranks, max ms over ranks)."""
    ms_max = max_over_ranks(ms_local, world, device)
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12, ms_max


def cpu_oracle_sample(w, q, k, v, target_s: float, seed: int = 0, threads: int | None = None,
                      num_targets=None, norm_gate=None, rab=None, candidates_only: bool = False):
    """Time the oracle on a bounded, uniformly random sample of rows.

    With ``norm_gate`` = (u, gamma, beta, eps) the sample is of tokens, each
    with all its heads and the output stage.  With ``candidates_only`` the
    rows are drawn from the candidates' rows.
    Returns (flops_of_sample / seconds, description, threads, seconds)."""
    from oracle import reference
    threads = threads or reference.default_threads()
    rng = np.random.default_rng(seed)
    off = w.offsets.astype(np.int64)
    seq_of = np.repeat(np.arange(w.batch), w.lengths)
    hist_of = (w.lengths - (np.asarray(num_targets, dtype=np.int64) if num_targets is not None
                            else 0)).astype(np.int64)

    per_row = w.heads if norm_gate is not None else 1

    pool = None
    if candidates_only:
        pool = np.concatenate([np.arange(off[b] + hist_of[b], off[b + 1]) for b in range(w.batch)])

    def rows(nr):
        nr = max(1, nr // per_row)
        t = rng.integers(0, w.total, size=nr) if pool is None else pool[rng.integers(0, len(pool), nr)]
        h = rng.integers(0, w.heads, size=nr)
        i = t - off[seq_of[t]]
        hist = hist_of[seq_of[t]]
        kept = np.where(i < hist, i + 1, hist + 1)
        return t, h, float(np.sum(4.0 * w.d * per_row * kept))

    def oracle(t, h):
        if norm_gate is not None:
            u, g, b, eps = norm_gate
            reference.hstu_rows_norm_gate(q, k, v, u, g, b, eps, w.offsets, w.alpha, w.inv_n, t,
                                          threads=threads, num_targets=num_targets, rab=rab)
        else:
            reference.hstu_rows(q, k, v, w.offsets, w.alpha, w.inv_n, t, h, threads=threads,
                                num_targets=num_targets, rab=rab)

    # calibrate on a small sample, then size the real one to ~target_s
    t, h, fl = rows(64)
    t0 = time.perf_counter()
    oracle(t, h)
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(max(64, min(2_000_000, 64 * target_s / dt)))
    t, h, fl = rows(n)
    t0 = time.perf_counter()
    oracle(t, h)
    dt = time.perf_counter() - t0
    if norm_gate is not None:
        desc = (f"{len(t)} uniformly sampled tokens (all {w.heads} heads, then the output stage) "
                f"of the {w.name} workload ({fl / 1e9:.2f} causal GFLOP), fp64 C oracle, "
                f"{threads} threads")
    else:
        desc = (f"{n} uniformly sampled (token, head) output rows "
                f"{'(candidates only) ' if candidates_only else ''}of the {w.name} workload "
                f"({fl / 1e9:.2f} causal GFLOP), fp64 C oracle, {threads} threads")
    return fl / dt / 1e12, desc, threads, dt


def run_reference_bwd(args, w, nt=None):
    world, rank, _ = dist_init()
    if rank != 0:
        return 0
    q, k, v = workloads.draw_qkv(w)
    rng = np.random.default_rng(4000 + max(w.index, 0))
    do = workloads.bf16_round(rng.standard_normal(q.shape).astype(np.float32))
    arrs = [t.float().numpy() for t in (q, k, v, do)]
    per_step_s = max(1.0, min(8.0, 150.0 / max(args.steps + args.warmup, 1)))
    vals = []
    desc, threads = "", 0
    for s_ in range(args.warmup + args.steps):
        val, desc, threads, _ = cpu_oracle_bwd_sample(w, *arrs, per_step_s, rab=_cpu_rab(args, w),
                                                      num_targets=nt)
        if s_ >= args.warmup:
            vals.append(val)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **w.describe(), "pass": "backward", **_targets_desc(nt),
                   **_rab_desc(args)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _norm_gate_desc(args) -> dict:
    if not args.norm_gate:
        return {}
    return {"output_stage": "Norm(A V) * U: layer norm over heads*d, affine gamma/beta, "
                            f"eps {workloads.NORM_EPS:g}, times U (HSTU paper section 3)"}


def _rab_desc(args) -> dict:
    if not args.rab:
        return {}
    return {"rab": "relative attention bias rab_{p,t}: log2-bucketed position and time tables, "
                   f"{workloads.RAB_BUCKETS} entries each (HSTU paper section 3)"}


def _cpu_rab(args, w):
    return workloads.draw_rab(w) if args.rab else None


def _cpu_norm_gate(args, w):
    if not args.norm_gate:
        return None
    u, g, b = workloads.draw_norm_gate(w)
    return u.float().numpy(), g, b, workloads.NORM_EPS


def run_reference(args, w, nt=None):
    world, rank, _ = dist_init()
    if rank != 0:
        return 0
    q, k, v = workloads.draw_qkv(w)
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    ng = _cpu_norm_gate(args, w)
    per_step_s = max(1.0, min(8.0, 150.0 / max(args.steps + args.warmup, 1)))
    vals = []
    desc, threads = "", 0
    for s in range(args.warmup + args.steps):
        val, desc, threads, dt = cpu_oracle_sample(w, qf, kf, vf, per_step_s, seed=s,
                                                   num_targets=nt, norm_gate=ng, rab=_cpu_rab(args, w),
                                                   candidates_only=args.candidates_only)
        if s >= args.warmup:
            vals.append(val)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **w.describe(), **_targets_desc(nt), **_norm_gate_desc(args),
                   **_rab_desc(args), **_co_desc(args)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _co_desc(args) -> dict:
    if not args.candidates_only:
        return {}
    return {"rows": "the candidates' only (HSTU_PLAN_CANDIDATES_ONLY): the history's keys and "
                    "values are a resident cache"}


def _targets_desc(nt) -> dict:
    if nt is None:
        return {}
    return {"mask": "M-FALCON candidates (HSTU paper Appendix H)",
            "num_targets_per_sequence": int(np.asarray(nt)[0]) if len(set(np.asarray(nt).tolist())) == 1
            else "varies"}


def run_ours_bwd(args, w, nt=None):
    """The backward on its own plan: kernel-only value, one-shot e2e with host buffers."""
    import torch
    from hstu_jagged_attention_gb300 import binding, build

    world, rank, local = dist_init()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    q_h, k_h, v_h = workloads.draw_qkv(w)
    rng = np.random.default_rng(4000 + max(w.index, 0))
    do_h = workloads.bf16_round(rng.standard_normal(q_h.shape).astype(np.float32))
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    grads = [torch.empty_like(q) for _ in range(3)]
    rab = tgrads = None
    if args.rab:
        # the timestamps are per-batch inputs (copied in every e2e step); the
        # tables are parameters, resident on the device
        rab_h = workloads.draw_rab(w)
        ts_pin = torch.from_numpy(rab_h[0]).pin_memory()
        rab = (ts_pin.to(dev), torch.from_numpy(rab_h[1]).to(dev), torch.from_numpy(rab_h[2]).to(dev))
        tgrads = (torch.empty_like(rab[1]), torch.empty_like(rab[2]))
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                       binding.HSTU_PLAN_BACKWARD)

    def plan_call():
        if rab is None:
            binding.hstu_attn_bwd_plan(plan, q, k, v, do, w.alpha, w.inv_n, *grads, stream=stream)
        else:
            binding.hstu_attn_bwd_plan_ex(plan, q, k, v, do, w.alpha, w.inv_n, *grads, rab=rab,
                                          dpos=tgrads[0], dtime=tgrads[1], stream=stream)

    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local)
    t_warm = time.perf_counter()
    for _ in range(args.warmup):
        plan_call()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        plan_call()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop(wall0, wall0 + wall, t_warm)
    times_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = statistics.mean(times_ms)
    flops = bwd_flops(w, nt)
    value, ms_max = aggregate(flops, ms, world, dev)
    st, site = binding.hstu_last_status()
    if st != binding.HSTU_OK:
        raise RuntimeError(f"device wait gave up during the timed region (site {site})")
    # end to end: host inputs in, gradients out, through the one-shot call
    pin = [t.pin_memory() for t in (q_h, k_h, v_h, do_h)]
    outs_h = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(3)]
    ins = [torch.empty_like(q) for _ in range(4)]
    g2 = [torch.empty_like(q) for _ in range(3)]
    offsets_host = w.offsets.copy()
    if rab is not None:
        tse = torch.empty_like(rab[0])
        tg_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in tgrads]
        tg2 = [torch.empty_like(t) for t in tgrads]

    def e2e_step():
        for dst, src in zip(ins, pin):
            dst.copy_(src, non_blocking=True)
        if rab is None and nt is None:
            binding.hstu_attn_bwd(*ins, offsets_host, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                  w.inv_n, *g2, stream=stream)
        elif rab is None:
            binding.hstu_attn_bwd_ex(*ins, offsets_host, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                     w.inv_n, *g2, num_targets=nt, stream=stream)
        else:
            tse.copy_(ts_pin, non_blocking=True)
            binding.hstu_attn_bwd_ex(*ins, offsets_host, w.batch, w.heads, w.d, w.max_seqlen, w.alpha,
                                     w.inv_n, *g2, num_targets=nt, rab=(tse, rab[1], rab[2]),
                                     dpos=tg2[0], dtime=tg2[1], stream=stream)
            for dst, src in zip(tg_h, tg2):
                dst.copy_(src, non_blocking=True)
        for dst, src in zip(outs_h, g2):
            dst.copy_(src, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        flush.zero_()
        e2e_step()
    e1.record(stream)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        flush.zero_()
    f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max(e0.elapsed_time(e1) / args.steps - f0.elapsed_time(f1) / args.steps, 1e-6)
    e2e_value, e2e_ms = aggregate(flops, e2e_ms, world, dev)
    elem = w.total * w.heads * w.d * 2
    h2d_extra = 0 if rab is None else int(ts_pin.numel() * ts_pin.element_size())
    d2h_extra = 0 if rab is None else int(sum(t.numel() * t.element_size() for t in tgrads))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        arrs = [t.float().numpy() for t in (q_h, k_h, v_h, do_h)]
        val, desc, threads, _ = cpu_oracle_bwd_sample(w, *arrs, args.cpu_seconds, rab=_cpu_rab(args, w),
                                                      num_targets=nt)
        cpu = {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}
    binding.hstu_plan_destroy(plan)
    peaks = load_peaks()
    achieved = flops / (ms * 1e-3) / 1e12
    if rank == 0:
        line = {
            "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**w.describe(), "pass": "backward", **_targets_desc(nt), **_rab_desc(args),
                       "l2": "flushed between steps (256 MiB write)",
                       "work_items": len(binding.hstu_worklist_build_bwd(w.offsets, w.heads)),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_bf16_peak": 100.0 * achieved / peaks["bf16_tflops"],
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                         "unit": UNIT, "frac": achieved / peaks["bf16_tflops"], "traffic": None,
                         "peak_source": f"{peaks['source']} bf16_tflops (burst)"},
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": 4 * elem + offsets_host.nbytes + h2d_extra,
                    "d2h_bytes_per_step": 3 * elem + d2h_extra, "ms_per_step": e2e_ms},
            "cpu_baseline": cpu,
            # the backward kernel and the dQ conversion per step
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
            "timed_wall_s": wall,
            "ms_per_step_min": min(times_ms),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_ours(args, w, nt=None):
    import torch
    from hstu_jagged_attention_gb300 import binding, build

    world, rank, local = dist_init()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build.build()

    q_h, k_h, v_h = workloads.draw_qkv(w)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    out = torch.empty_like(q)
    ng = args.norm_gate
    if ng:
        # gamma and beta are the layer's weights: resident on the device
        u_h, g_h, b_h = workloads.draw_norm_gate(w)
        u = u_h.to(dev)
        gamma, beta = torch.from_numpy(g_h).to(dev), torch.from_numpy(b_h).to(dev)
        eps = workloads.NORM_EPS
    rab = None
    if args.rab:
        # the tables are weights, resident on the device; the timestamps are
        # per-token inputs
        ts_h, pos_h, time_h = workloads.draw_rab(w)
        ts_pin = torch.from_numpy(ts_h).pin_memory()
        rab = (ts_pin.to(dev), torch.from_numpy(pos_h).to(dev), torch.from_numpy(time_h).to(dev))
    co = args.candidates_only
    if co and (nt is None or ng):
        raise SystemExit("--candidates-only needs the candidates workload and no --norm-gate")
    plan = binding.hstu_plan_create_ex(w.offsets, nt, w.batch, w.heads, w.d, w.max_seqlen,
                                       (binding.HSTU_PLAN_NORM_GATE if ng else 0) |
                                       (binding.HSTU_PLAN_CANDIDATES_ONLY if co else 0))

    def launch():
        binding.hstu_attn_fwd_plan_ex(plan, q, k, v, w.alpha, w.inv_n, out, rab=rab,
                                      norm_gate=(u, gamma, beta, eps) if ng else None, stream=stream)

    n_items = binding.hstu_plan_num_items(plan)
    grid, block, smem = binding.hstu_launch_shape(plan)
    if ng:
        block = 512  # two SiLU warpgroups (the shape query assumes no output stage)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)

    sampler = ClockSampler(local)
    t_warm = time.perf_counter()
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize(dev)
    st, site = binding.hstu_last_status()
    if st != binding.HSTU_OK:
        raise RuntimeError(f"device wait gave up during warm-up (site {site})")

    # ---- kernel-only timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(wall0, wall0 + wall, t_warm)
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = statistics.mean(times_ms)
    flops = candidate_row_flops(w, nt) if co else causal_flops(w, nt)
    value, ms_max = aggregate(flops, ms, world, dev)
    st, site = binding.hstu_last_status()
    if st != binding.HSTU_OK:
        raise RuntimeError(f"device wait gave up during the timed region (site {site})")

    peaks = load_peaks()
    peak = peaks["bf16_tflops"]
    achieved = flops / (ms * 1e-3) / 1e12
    traffic = None
    key = w.name + ("+norm_gate" if ng else "") + ("+rab" if args.rab else "")
    if MEASURED_TRAFFIC.get(key) and MEASURED_TRAFFIC.get("sha256") == kernel_sha():
        traffic = MEASURED_TRAFFIC[key]

    # ---- end to end through the C ABI with host buffers
    pin = [t.pin_memory() for t in ((q_h, k_h, v_h, u_h) if ng else (q_h, k_h, v_h))]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    qe, ke, ve, ue = (torch.empty_like(q) for _ in range(4))
    oe = torch.empty_like(out)
    offsets_host = w.offsets.copy()

    tse = torch.empty_like(rab[0]) if rab is not None else None
    # candidates only: the history's keys and values (and queries) are the
    # resident cache; each step brings the candidates' q, k, v rows and
    # returns their outputs, one copy per sequence and tensor
    cand_rows = []
    if co:
        for dst, src in zip((qe, ke, ve), pin[:3]):
            dst.copy_(src)
        off = w.offsets.astype(np.int64)
        cand_rows = [(int(off[b + 1] - nt[b]), int(off[b + 1])) for b in range(w.batch) if nt[b] > 0]

    def e2e_step_candidates():
        for s0, s1 in cand_rows:
            qe[s0:s1].copy_(pin[0][s0:s1], non_blocking=True)
            ke[s0:s1].copy_(pin[1][s0:s1], non_blocking=True)
            ve[s0:s1].copy_(pin[2][s0:s1], non_blocking=True)
        binding.hstu_attn_fwd_plan_ex(plan, qe, ke, ve, w.alpha, w.inv_n, oe,
                                      rab=(tse, rab[1], rab[2]) if rab is not None else None,
                                      stream=stream)
        for s0, s1 in cand_rows:
            out_h[s0:s1].copy_(oe[s0:s1], non_blocking=True)

    def e2e_step():
        if co:
            if rab is not None:
                tse.copy_(ts_pin, non_blocking=True)
            e2e_step_candidates()
            return
        if nt is None and not ng and rab is None:
            # host buffers in and out through the library's chunked call, its
            # copies overlapped with the kernel
            binding.hstu_attn_fwd_host(pin[0], pin[1], pin[2], offsets_host, w.batch, w.heads, w.d,
                                       w.max_seqlen, w.alpha, w.inv_n, out_h, qe, ke, ve, oe,
                                       stream=stream)
            return
        qe.copy_(pin[0], non_blocking=True)
        ke.copy_(pin[1], non_blocking=True)
        ve.copy_(pin[2], non_blocking=True)
        if ng:
            ue.copy_(pin[3], non_blocking=True)
        if rab is not None:
            tse.copy_(ts_pin, non_blocking=True)
        if ng or rab is not None:
            binding.hstu_attn_fwd_ex(qe, ke, ve, offsets_host, w.batch, w.heads, w.d, w.max_seqlen,
                                     w.alpha, w.inv_n, oe, num_targets=nt,
                                     rab=(tse, rab[1], rab[2]) if rab is not None else None,
                                     norm_gate=(ue, gamma, beta, eps) if ng else None, stream=stream)
        elif nt is None:
            binding.hstu_attn_fwd(qe, ke, ve, offsets_host, w.batch, w.heads, w.d, w.max_seqlen,
                                  w.alpha, w.inv_n, oe, stream)
        else:
            binding.hstu_attn_fwd_targets(qe, ke, ve, offsets_host, nt, w.batch, w.heads, w.d,
                                          w.max_seqlen, w.alpha, w.inv_n, oe, stream)
        out_h.copy_(oe, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    for _ in range(args.steps):
        flush.zero_()  # same L2 state as the kernel-only region
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    flush_ms = 0.0
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        flush.zero_()
    f1.record(stream)
    torch.cuda.synchronize(dev)
    flush_ms = f0.elapsed_time(f1) / args.steps
    e2e_ms = max(e0.elapsed_time(e1) / args.steps - flush_ms, 1e-6)
    e2e_value, e2e_ms = aggregate(flops, e2e_ms, world, dev)
    st, site = binding.hstu_last_status()
    if st != binding.HSTU_OK:
        raise RuntimeError(f"device wait gave up during the e2e region (site {site})")
    elem = 2
    h2d = (4 if ng else 3) * w.total * w.heads * w.d * elem + offsets_host.nbytes
    if rab is not None:
        h2d += 4 * w.total
    d2h = w.total * w.heads * w.d * elem
    if co:
        n_cand = sum(s1 - s0 for s0, s1 in cand_rows)
        h2d = 3 * n_cand * w.heads * w.d * elem + (4 * w.total if rab is not None else 0)
        d2h = n_cand * w.heads * w.d * elem

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qf, kf, vf = (t.float().numpy() for t in (q_h, k_h, v_h))
        val, desc, threads, _ = cpu_oracle_sample(w, qf, kf, vf, args.cpu_seconds, num_targets=nt,
                                                  norm_gate=_cpu_norm_gate(args, w),
                                                  rab=_cpu_rab(args, w), candidates_only=co)
        cpu = {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}

    binding.hstu_plan_destroy(plan)
    per_config = cpu_st = None
    if (rank == 0 and world == 1 and not args.no_per_config and not (ng or args.rab or co)
            and nt is None and not args.sweep):
        per_config = per_config_report(dev, stream, flush, args.steps, args.warmup, peaks)
        if not args.no_cpu_baseline:
            cpu_st = cpu_single_thread_report(args.cpu_single_seconds)
    roof = roofline_entry(flops, algorithmic_bytes(w, ng), ms, peaks)
    bound = roof["bound"]
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**w.describe(), **_targets_desc(nt), **_norm_gate_desc(args), **_rab_desc(args),
                       **_co_desc(args),
                       "l2": "flushed between steps (256 MiB write)",
                       "work_items": n_items, "grid": grid, "block": block, "smem_bytes": smem,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_bf16_peak": 100.0 * achieved / peak,
            "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                          "frac": achieved / peak, "traffic": traffic,
                          "peak_source": f"{peaks['source']} bf16_tflops (burst)",
                          "algorithmic_bytes": algorithmic_bytes(w, ng),
                          "flop_per_byte": roof["flop_per_byte"], "ridge_flop_per_byte": roof["ridge_flop_per_byte"]}
                         if bound == "tensor" else
                         {"bound": "hbm", "achieved": roof["hbm_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": roof["hbm_gbs"] / peaks["hbm_gbs"], "traffic": traffic,
                          "peak_source": f"{peaks['source']} hbm_gbs",
                          "algorithmic_bytes": algorithmic_bytes(w, ng),
                          "flop_per_byte": roof["flop_per_byte"], "ridge_flop_per_byte": roof["ridge_flop_per_byte"]}),
            "hbm_gbs": roof["hbm_gbs"], "pct_of_hbm_peak": roof["pct_of_hbm_peak"],
            "per_config": per_config,
            "cpu_baseline_single_thread": cpu_st,
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "call": ("hstu_attn_fwd_host (runs of sequences, copies overlapped with the kernel)"
                             if nt is None and not ng and rab is None else
                             "copies in, one-shot call, copy out, on one stream")},
            "cpu_baseline": cpu,
            # the attention kernel per step, and the output-stage kernel after it
            # (the per-config timings run outside the timed region)
            "gpu_launches": args.steps * (2 if ng else 1),
            "clocks": clocks,
            "timed_wall_s": wall,
            "ms_per_step_min": min(times_ms),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(workloads.WORKLOAD_NAMES) + ["candidates"],
                    default="dense")
    ap.add_argument("--sweep", action="store_true", help="one line per workload (extra lines)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-single-seconds", type=float, default=6.0,
                    help="seconds of single-thread oracle work on the dense workload")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config timings of the five workloads")
    ap.add_argument("--norm-gate", action="store_true",
                    help="fuse the layer's output stage Norm(A V) * U into the timed call")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (dQ, dK, dV) instead of the forward")
    ap.add_argument("--candidates-only", action="store_true",
                    help="with --workload candidates: compute the candidates' rows only "
                         "(the history's keys and values cached)")
    ap.add_argument("--rab", action="store_true",
                    help="add the relative attention bias rab_{p,t} (timestamps and bucketed tables)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.candidates_only and (args.workload != "candidates" or args.backward or args.sweep
                                 or args.norm_gate):
        ap.error("--candidates-only goes with --workload candidates (forward, no --norm-gate)")
    names = list(workloads.WORKLOAD_NAMES) + ["candidates"] if args.sweep else [args.workload]
    rc = 0
    for name in names:
        w, nt = workload_by_name(name)
        if args.backward:
            rc |= run_reference_bwd(args, w, nt) if args.impl == "reference" else run_ours_bwd(args, w, nt)
        else:
            rc |= run_reference(args, w, nt) if args.impl == "reference" else run_ours(args, w, nt)
    return rc


if __name__ == "__main__":
    sys.exit(main())
