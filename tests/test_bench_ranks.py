"""Multi-rank logic of bench.py on CPU: world size 2 over gloo.

Each rank runs the same workload (weak scaling, no data-path collective);
the job time is the slowest rank's and the throughput counts every rank's
work.  The ranks here report different times; both must agree on the max.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_init() == (world, rank, rank)
    ms_local = 2.0 if rank == 0 else 5.0
    value, ms_max = bench.aggregate(1e12, ms_local, world)
    results[rank] = (value, ms_max)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs)
        res = dict(results)
    # both ranks see the max time (5 ms); 2 ranks x 1e12 FLOP in 5 ms = 400 TFLOP/s
    for r in range(world):
        value, ms_max = res[r]
        assert ms_max == 5.0
        assert value == pytest.approx(400.0)


def test_single_rank_aggregation_needs_no_process_group():
    import bench
    value, ms = bench.aggregate(2e12, 4.0, 1)
    assert ms == 4.0 and value == pytest.approx(500.0)


@pytest.mark.parametrize("extra", [[], ["--backward"], ["--workload", "candidates", "--candidates-only"]])
def test_reference_arm_runs_on_rank_zero_only(extra):
    # under torchrun every rank but 0 exits at once, prints nothing and
    # touches the oracle not at all
    import subprocess
    import sys
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3", *extra],
                       env=env, capture_output=True, text=True, timeout=120, cwd=root)
    assert r.returncode == 0, r.stderr[-500:]
    assert r.stdout.strip() == ""
