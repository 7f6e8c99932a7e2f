"""The bench's multi-process path on the CPU (gloo, world size 2): replicas time independently and
rank 0 reports the slowest rank's time; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        # each rank's own elapsed time; every rank must get the slowest one
        t = bench.barrier_max(0.25 * (rank + 1), 2)
        bench.barrier(2)
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_reaches_every_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(_free_port(), out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: 0.5, 1: 0.5}


def test_single_process_keeps_its_own_time():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.barrier_max(1.25, 1) == 1.25
    bench.barrier(1)  # no process group: nothing to wait for


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import argparse

    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.reference_arm(argparse.Namespace(steps=1, warmup=0))
    assert capsys.readouterr().out == ""  # the other ranks exit without work or output
