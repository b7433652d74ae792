"""The N > 1 path of bench.py on CPU: world-size-2 gloo process groups.

The codec has no exchange step, so several GPUs run independent replicas;
what crosses ranks is only the bench's timing: a barrier around the timed
region and the maximum of the per-rank step times.  These tests run that
code as two gloo ranks on 127.0.0.1 (no GPU), and check that the reference
arm lets rank 1 exit without work.
"""
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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    step_ms = 1.5 + rank  # rank 1 is the slower one
    slowest = bench.max_over_ranks(dist, step_ms, "cpu")
    bench.barrier(dist)
    q.put((rank, slowest))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}  # every rank sees the slowest rank's time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.25, "cpu") == 3.25
    bench.barrier(None)


def test_reference_arm_rank1_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("world", [1, 2, 4])
def test_weak_scaling_value_counts_every_rank(world):
    """value = units all ranks processed / the slowest rank's time."""
    sys.path.insert(0, ROOT)
    import bench
    step_bytes, ms = 2 * 2 * 58_720_256, 0.1
    assert bench.aggregate_gbs(world, step_bytes, ms) == pytest.approx(world * step_bytes / (ms * 1e-3) / 1e9)
