"""The benchmark's multi-rank path on CPU (gloo, world size 2).

With --gpus N the GEMV runs as N independent replicas (the path has no exchange step): every
rank times the same workload on its own GPU, the job time is the slowest rank's (an all-reduce
MAX) and the value is all ranks' bytes over it.  These tests run that host logic on CPU ranks.
"""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_dist(world, "gloo")
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        bench.barrier(world)
        seconds = 1.0 + 0.5 * rank                 # rank 1 is the slower one
        job = bench.max_over_ranks(seconds, world)  # CPU tensors under gloo
        bench.barrier(world)
        out.put((rank, job, bench.job_throughput_gbps(world, 10, 2 * 10 ** 9, job)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get(timeout=5) for _ in range(2))
    # both ranks see the max (1.5 s); the value counts both ranks' bytes: 2 * 10 * 2 GB / 1.5 s
    assert [g[1] for g in got] == [1.5, 1.5]
    assert all(abs(g[2] - 2 * 10 * 2 / 1.5) < 1e-9 for g in got)


def test_reference_arm_on_a_non_zero_rank_exits_without_work():
    """Under torchrun only rank 0 runs and prints the reference arm; the others exit 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
