"""Multi-rank host logic on the CPU (gloo, world size 2).

The path shards with no data exchange (independent replicas, weak scaling);
bench.py only needs a max over ranks for time and a sum for work, and the
reference arm runs on rank 0 alone.  These run as CPU processes."""

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
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    t = 10.0 + rank          # per-rank elapsed time
    work = 100.0 * (rank + 1)  # per-rank units
    mx = bench.allreduce(t, world, "cpu", "max")
    sm = bench.allreduce(work, world, "cpu", "sum")
    bench.barrier(world)
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn",
                       join=True)
    for r in range(world):
        mx, sm = out[r]
        assert mx == 11.0          # the job time is the slowest rank's
        assert sm == 300.0         # whole-job work is the sum over ranks


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_gpus_flag_must_match_the_launch():
    """--gpus N without N ranks is refused instead of silently running one."""
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--steps", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE" in (r.stderr + r.stdout)
