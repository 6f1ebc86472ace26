"""Host logic of the multi-GPU benchmark path on CPU: gloo ranks, no GPU.

bench.py runs one independent replica per GPU (sequences never interact, so
there is no data-path collective); the job's time is the slowest rank's and
its throughput counts every rank's units.  These tests run that aggregation
on two gloo processes, and check that the reference arm's extra ranks exit
cleanly without work.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [3.0, 7.5][rank]
        slowest = bench.max_over_ranks(ms, torch.device("cpu"), world)
        gbs = bench.job_throughput(1e9, slowest / 1e3, world) / 1e9
        dist.barrier()
        out[rank] = (slowest, gbs)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slowest, gbs = res[r]
        assert slowest == 7.5                                   # every rank sees the max
        assert gbs == pytest.approx(2 * 1e9 / 7.5e-3 / 1e9)      # both ranks' bytes / max time


def test_single_rank_aggregation_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, torch.device("cpu"), 1) == 4.25
    assert bench.job_throughput(10.0, 2.0, 1) == 5.0


def test_reference_arm_extra_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
