"""Host logic of the multi-GPU bench run (replicas, weak scaling), exercised
with world-size-2 gloo ranks on the CPU: the timing reduction takes the
slowest rank, the whole-job rate counts every rank's batch, every rank gets
its own batch, and the reference arm does its work on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = (bench.max_over_ranks(times[rank]), bench.rank_seed(rank))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_time():
    world, port = 2, _free_port()
    times = [0.125, 0.5]
    # spawn, not fork: earlier tests may have started threads in this process
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == max(times)
    assert res[0][1] != res[1][1]  # every rank verifies its own batch


def test_whole_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job_rate(1792, 1, 0.5e-3) == pytest.approx(1792 / 0.5e-3)
    assert bench.whole_job_rate(1792, 4, 0.5e-3) == pytest.approx(4 * 1792 / 0.5e-3)
    assert bench.max_over_ranks(0.25) == 0.25  # no process group: the value itself


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
