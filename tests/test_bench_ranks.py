"""The benchmark's multi-rank host logic on CPU processes (gloo, world size 2, 127.0.0.1).

The path shards into independent replicas (no collective on the data path); the only exchange
is the timing reduction: each reported time is the slowest rank's, and only rank 0 prints the
reference arm."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0 * rank], dist, "cpu")
        alone = bench.max_over_ranks([1.0 + rank])
        silent = bench.run_reference(None, rank, world) if rank != 0 else None
        q.put((rank, got, alone, silent))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank0_only_reference():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, alone, silent in out:
        assert got == [2.0, 10.0, 5.0]          # element-wise max over both ranks
        assert alone == [1.0 + rank]           # one process: its own values
        assert silent is None                  # rank 1 does no reference work
