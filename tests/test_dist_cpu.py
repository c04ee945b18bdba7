"""The multi-rank path of bench.py on CPU: world size 2 over gloo (127.0.0.1).
Each rank runs its own shard of the workload (weak scaling, no data exchange);
the only collective is the max-over-ranks timing reduction."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from sparse_attention_layout_gb300 import workloads as W
    ms = bench.max_over_ranks(10.0 + rank, world, "cpu")  # rank 1 is the slow one
    value = bench.weak_value(1.0e12, world, ms)
    q, _, _ = W.TINY.qkv(shard=rank)
    gathered = [torch.zeros_like(q) for _ in range(world)]
    dist.all_gather(gathered, q)  # test-side only: compare the shards
    out[rank] = (ms, value, bool(torch.equal(gathered[0], gathered[1])),
                 bool(torch.equal(q, W.TINY.qkv(shard=rank)[0])))
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for rank in range(world):
        ms, value, same_shards, reproducible = out[rank]
        assert ms == pytest.approx(11.0)                  # max over ranks
        assert value == pytest.approx(2.0e12 / 11.0e-3 / 1e12)  # both ranks' work / slowest time
        assert not same_shards                            # each rank draws its own batch
        assert reproducible                               # seeded
