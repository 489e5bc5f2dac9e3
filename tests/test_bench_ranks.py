"""bench.py's multi-rank accounting on the CPU: two gloo ranks, each timing
its own replica; the job reports the slowest rank's time and the summed
iterations (the path has no collective of its own)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.0, 150.0][rank]
    iters = [37, 38][rank]
    res = bench.reduce_over_ranks(ms, iters, torch.device("cpu"))
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_takes_max_time_and_summed_work():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == out[1] == (150.0, 75.0)


def test_single_process_is_identity():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(12.5, 7, torch.device("cpu")) == (12.5, 7.0)
