"""The N > 1 path of the benchmark on CPU: replicas only (no data-path collective).

Two gloo ranks on 127.0.0.1 stand in for two GPUs: the whole-job time is the
slowest rank's, the throughput counts every rank's units, and the reference arm
runs on rank 0 only (the other ranks exit 0 without work).
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


def _rank_main(rank, world, port, times, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    t, v = bench.replica_totals(times[rank], 1000, world, dist, torch.device("cpu"))
    out[rank] = (t, v)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.5, 2.0), (3.0, 1.0)])
def test_replica_totals_two_gloo_ranks(times):
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
        got = dict(out)
    slowest = max(times)
    for r in range(world):
        t, v = got[r]
        assert t == slowest
        assert v == pytest.approx(world * 1000 / slowest)


def test_replica_totals_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_totals(0.25, 1000, 1) == (0.25, 4000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
