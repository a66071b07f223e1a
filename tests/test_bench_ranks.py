"""bench.py's multi-rank bookkeeping on the CPU: two gloo ranks (127.0.0.1)
reduce their timings to the slowest and report the same whole-job value; the
reference arm runs on rank 0 only.  No GPU is touched."""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_ms, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(local_ms[rank], dist, "cpu")
    out[rank] = (slowest, bench.job_tflops(world, 10, 2e12, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest():
    world, port = 2, _free_port()
    local_ms = [120.0, 150.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, local_ms, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, value = res[0]
    assert slowest == 150.0
    assert value == pytest.approx(2 * 10 * 2e12 / 0.150 / 1e12)


def test_single_rank_is_its_own_maximum():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1, 4, 1e12, 1000.0) == pytest.approx(4.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0
    assert res.stdout.strip() == ""
