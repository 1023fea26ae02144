"""Host logic of the multi-rank benchmark, on CPU with the gloo backend.

Each rank of a ``bench.py --gpus N`` run times its own sequences (no data
exchange on the path); the job's time is the slowest rank's and its
throughput counts every rank's units.  Two gloo ranks on CPU check that
reduction without a GPU.
"""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total, value = bench.aggregate_over_ranks(10.0 * (rank + 1), units_per_rank=8, steps=5, world=world,
                                              device="cpu")
    out[rank] = (total, value)
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        total, value = out[rank]
        assert total == 20.0                       # the slowest rank's time
        assert value == world * 8 * 5 / 0.020      # every rank's units over that time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_over_ranks(4.0, 8, 2, 1, "cpu") == (4.0, 8 * 2 / 0.004)
