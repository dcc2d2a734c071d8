"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): the
barrier and the max-over-ranks timing reduction, and the weak-scaling
throughput that counts every rank's tokens."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
    out[rank] = ms
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
