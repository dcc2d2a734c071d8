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


def _shard_rank_main(rank, world, port, out):
    """One rank of a --shard bh run on CPU: it takes its (b, h) slice with
    bench.shard_bh / bench.shard_inputs and scans it with the oracle (called
    here, by the test: bench.py never runs the oracle on this path)."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import ttm_inputs as wl
    w, inp = wl.generate_custom(kind="titans", dtype="f32", B=3, H=5, T=40, d=8, chunk=16,
                                w0_shared=True, seed=3)
    lo, hi = bench.shard_bh(w.B, w.H, rank, world)
    ws, sub = bench.shard_inputs(w, inp, lo, hi)
    f = lambda t: None if t is None else t.double().numpy()
    r = oracle.linear_primal(f(sub["q"]), f(sub["k"]), f(sub["v"]), f(sub["theta"]), f(sub["W0"]),
                             ws.chunk, eta=f(sub["eta"]), alpha=f(sub["alpha"]), threads=1)
    parts = [None] * world
    dist.all_gather_object(parts, (lo, hi, r["z"][0], r["W"][0], r["S"][0]))
    if rank == 0:
        out["parts"] = parts
    dist.destroy_process_group()


def test_bh_shard_two_gloo_ranks_cover_every_sequence_once():
    import numpy as np

    import oracle
    import ttm_inputs as wl
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_shard_rank_main, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    parts = sorted(out["parts"], key=lambda p: p[0])
    w, inp = wl.generate_custom(kind="titans", dtype="f32", B=3, H=5, T=40, d=8, chunk=16,
                                w0_shared=True, seed=3)
    units = [u for lo, hi, *_ in parts for u in range(lo, hi)]
    assert units == list(range(w.B * w.H))              # every unit exactly once, in order
    f = lambda t: None if t is None else t.double().numpy()
    whole = oracle.linear_primal(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["theta"]),
                                 f(inp["W0"]), w.chunk, eta=f(inp["eta"]), alpha=f(inp["alpha"]),
                                 shared_over_batch=True, threads=1)
    for key, idx in (("z", 2), ("W", 3), ("S", 4)):
        cat = np.concatenate([p[idx] for p in parts], axis=0)
        assert np.array_equal(cat, whole[key].reshape(w.B * w.H, *whole[key].shape[2:])), key


def test_bh_shard_ranges_are_balanced():
    import bench
    for n_b, n_h, world in ((1, 16, 8), (3, 5, 4), (8, 12, 7), (1, 1, 3)):
        spans = [bench.shard_bh(n_b, n_h, r, world) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == n_b * n_h
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        sizes = [hi - lo for lo, hi in spans]
        assert max(sizes) - min(sizes) <= 1
