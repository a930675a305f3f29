"""Host-side logic of bench.py's multi-process (replica) path, on CPU with gloo.

Each GPU runs an independent replica of the step; the job's time is the slowest
rank's, and the job's throughput counts every replica's bytes.  The reference arm
runs on rank 0 only; other ranks exit without work.
"""
from __future__ import annotations

import importlib.util
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        got = b.max_over_ranks(times[rank], world)
        out[rank] = (got, b.job_gbs(1_000_000_000, 10, world, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world, port = 2, _free_port()
    times = [12.5, 20.0]                     # ms: rank 1 is the slow one
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 20.0
    # 2 replicas x 10 steps x 1 GB in 20 ms = 1000 GB/s, on every rank
    assert res[0][1] == pytest.approx(1000.0) and res[1][1] == pytest.approx(1000.0)


def test_single_rank_is_identity():
    b = _bench()
    assert b.max_over_ranks(7.25, 1) == 7.25
    assert b.job_gbs(2_000_000_000, 4, 1, 8.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
