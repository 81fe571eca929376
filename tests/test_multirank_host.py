"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2).

Each rank of a torchrun launch runs its own independent problem (replicas, no
data-path collective); the only cross-rank steps are the barriers around the
timed region and the max of the per-rank step times.  These tests run that
logic with two gloo ranks and no GPU.
"""

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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        step_ms = 1.25 + 0.5 * r              # rank 1 is the slower one
        m = bench.max_over_ranks(step_ms, w, torch.device("cpu"))
        value = bench.whole_job_rate(1000.0, w, m)
        bench.barrier(w)
        q.put((r, w, local, m, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    # Both ranks see the slowest rank's time; the job rate counts both ranks' units.
    assert res == [(0, 2, 0, 1.75, 2000.0 / 1.75e-3), (1, 2, 1, 1.75, 2000.0 / 1.75e-3)]


def test_whole_job_rate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(3.0, 1, 1.5) == pytest.approx(2000.0)
    assert bench.max_over_ranks(4.5, 1, None) == 4.5


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""
