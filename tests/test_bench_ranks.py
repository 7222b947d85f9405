"""Host logic of the multi-rank bench on CPU: two gloo ranks (no GPU).

Every rank runs its own replica of the step; the job's time per step is
the slowest rank's (an all-reduce MAX), and the job's rate counts every
rank's rows. The reference arm runs on rank 0 only.
"""

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 1.0 + 0.5 * rank  # rank 1 is the slow one
        ms = bench._max_over_ranks(local_ms, world, torch.device("cpu"))
        q.put((rank, ms, bench._job_rate(1000, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_and_count_all_rows():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in got:
        assert ms == pytest.approx(1.5)
        assert rate == pytest.approx(1000 * 2 / 1.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._max_over_ranks(2.5, 1, None) == 2.5
    assert bench._job_rate(20544, 1, 2.0) == pytest.approx(20544 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
