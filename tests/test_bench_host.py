"""Host-side logic of the multi-rank benchmark, on CPU ranks with gloo.

Each rank verifies its own batch (no collective on the data path); the only
collectives are the barrier and the max-over-ranks reduction of the step time,
and the whole-job rate is all ranks' units over the slowest rank's time."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d, r, ws = bench._dist()
    cpu = torch.device("cpu")
    try:
        bench._barrier(d, cpu)
        # rank r took (r + 1) ms for its step: the job time is the slowest rank's
        ms = bench._max_over_ranks(d, float(r + 1), cpu)
        rate = bench.job_rate(ws, 1000, ms)
        q.put((r, ws, ms, rate))
    finally:
        d.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(world))
    for r, (rank, ws, ms, rate) in enumerate(got):
        assert rank == r and ws == world
        assert ms == 2.0                       # the slowest rank's time
        assert rate == world * 1000 / 0.002    # all ranks' units / that time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(None, 3.5, torch.device("cpu")) == 3.5
    assert bench.job_rate(1, 64 * 16, 0.25) == 64 * 16 / 0.00025


@pytest.mark.skipif(not dist.is_gloo_available(), reason="needs gloo")
def test_reference_arm_under_torchrun_prints_one_line():
    """`bench.py --impl reference` launched like the multi-GPU bench: rank 0
    alone times the oracle and prints the line; the other rank exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "greedy_tiny", "--gpus", "2", "--steps", "2",
           "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the steps it timed (all of them here: the run fits its time budget)
    assert line["steps_requested"] == 2 and line["steps"] == 2 and line["warmup"] == 1
    # one sequence (greedy tiny has B = 1): one oracle thread had work
    assert line["cpu_baseline"]["cores"] == 1


def test_workload_launch_counts_and_tv_flag():
    """Library kernels per step that `gpu_launches` reports: the lenient sweep
    computes the per-row TV by default (one more kernel), --no-tv leaves it
    out; the other workloads are unchanged."""
    sys.path.insert(0, ROOT)
    import argparse
    import bench

    def args(**kw):
        d = dict(batch=None, T=None, sigma=None, lam=None, mode=None, no_tv=False)
        d.update(kw)
        return argparse.Namespace(**d)

    # a sampling call: streaming pass, residual pass (correction or bonus),
    # fp64 check (+ the TV pass)
    w = bench.Workload("lenient_sweep", args())
    assert w.tv and w.launches() == 4 and w.point()["tv"] is True
    w = bench.Workload("lenient_sweep", args(no_tv=True))
    assert not w.tv and w.launches() == 3 and w.point()["tv"] is False
    w = bench.Workload("lossless_t1", args())
    assert not w.tv and w.launches() == 3
    assert bench.Workload("tree", args(T=1.0)).launches() == 2
    assert bench.Workload("tree", args(T=0.0)).launches() == 1
    assert bench.Workload("packed", args(T=1.0)).launches() == 4
    assert bench.Workload("packed", args(T=0.0)).launches() == 1
    assert bench.Workload("spot", args(T=1.0)).launches() == 3
    assert bench.Workload("spot", args(T=0.0)).launches() == 2
    assert bench.Workload("anyorder", args()).launches() == 2
    assert bench.Workload("packed_topk", args()).launches() == 2
    assert bench.Workload("greedy_tiny", args()).launches() == 1
