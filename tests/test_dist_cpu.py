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


# ---------------------------------------------------- one workload split ----

def test_balanced_ranges_cover_every_pair_once_with_bounded_imbalance():
    import numpy as np
    from sparse_attention_layout_gb300 import partition, workloads as W
    layouts = [W.BIGBIRD.layout(), W.STRIDED.layout(), W.BAND.layout(),
               W.layout_random_diag(12, 0.3, H=7, seed=3), np.zeros((3, 4, 4), np.uint8)]
    for lay in layouts:
        for Z in (1, 2, 5):
            w = partition.pair_weights(lay, Z)
            for world in (1, 2, 3, 4, 8, 64):
                ranges = partition.balanced_ranges(w, world)
                assert len(ranges) == world
                covered = np.concatenate([np.arange(a, b) for a, b in ranges])
                assert np.array_equal(covered, np.arange(w.size))           # each pair exactly once, in order
                loads = [int(w[a:b].sum()) for a, b in ranges]
                assert max(loads) <= w.sum() / world + (w.max() if w.size else 0)


def _split_worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import numpy as np
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from sparse_attention_layout_gb300 import partition, workloads as W
    lay = W.layout_bigbird(8, H=3, seed=4)
    Z, B, D = 2, 16, 32
    S = 8 * B
    Q, K, V = (W.randn((Z, 3, S, D), "f32", 90 + s) for s in range(3))
    u0, u1, sub = partition.shard_layout(lay, Z, rank, world)
    # this rank's pairs as one call: batch 1, u1 - u0 heads
    part = [t.reshape(1, Z * 3, S, D)[:, u0:u1] for t in (Q, K, V)]
    O = oracle.Oracle().attention(sub, B, *part, 0.2, W.MASK_DIAG_CAUSAL) if u1 > u0 else \
        np.zeros((1, 0, S, D))
    bounds = [None] * world
    dist.all_gather_object(bounds, (u0, u1))   # test-side only: assemble the ranks' results
    outs = [None] * world
    dist.all_gather_object(outs, O)
    if rank == 0:
        full = oracle.Oracle().attention(lay, B, Q, K, V, 0.2, W.MASK_DIAG_CAUSAL).reshape(1, Z * 3, S, D)
        joined = np.concatenate(outs, axis=1)
        out["bounds"] = bounds
        out["equal"] = bool(np.array_equal(joined, full))
    dist.destroy_process_group()


def test_two_ranks_split_one_workload_gloo():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_split_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    (a0, a1), (b0, b1) = out["bounds"]
    assert a0 == 0 and a1 == b0 and b1 == 6 and 0 < a1 < 6   # both ranks work, no pair twice
    assert out["equal"]                                       # the pieces are the whole result, bit for bit


def test_line_shards_cover_every_block_once():
    import numpy as np
    from sparse_attention_layout_gb300 import partition, workloads as W
    for lay in (W.layout_random_diag(12, 0.3, H=3, seed=3), W.BIGBIRD.layout(), np.zeros((2, 4, 4), np.uint8)):
        for orient in (0, 1):
            w = partition.line_weights(lay, orient)
            for world in (1, 2, 3, 8):
                ids, loads, prev = [], [], 0
                for r in range(world):
                    l0, l1, sub, kept = partition.shard_lines(lay, orient, r, world)
                    assert l0 == prev and l1 >= l0                     # contiguous lines, in order
                    prev = l1
                    assert sub.shape == lay.shape and int(sub.sum()) == kept.size
                    assert np.all(sub <= lay)                          # only the layout's own blocks
                    ids.append(kept)
                    loads.append(kept.size)
                assert prev == w.size
                assert np.array_equal(np.sort(np.concatenate(ids)), np.arange(int(lay.sum())))
                assert max(loads) <= w.sum() / world + (w.max() if w.size else 0)


def _spmm_split_worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import numpy as np
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from sparse_attention_layout_gb300 import partition, workloads as W
    orc = oracle.Oracle()
    lay = W.layout_random_diag(10, 0.35, H=2, seed=7)
    Z, B, N = 2, 16, 24
    S = 10 * B
    nnz = int(lay.sum())
    Asp = W.uniform((Z, nnz, B, B), "f32", 70)
    Bd = W.uniform((Z, 2, S, N), "f32", 71)
    Ad = W.uniform((Z, 2, N, S), "f32", 72)
    res = {}
    for orient, name in ((0, "dsd"), (1, "dds")):
        _, _, sub, ids = partition.shard_lines(lay, orient, rank, world)
        part = Asp[:, ids]
        C = orc.dsd(sub, B, part, Bd) if orient == 0 else orc.dds(sub, B, Ad, part)
        pieces = [None] * world
        dist.all_gather_object(pieces, C)   # test-side only: assemble the ranks' disjoint outputs
        if rank == 0:
            full = orc.dsd(lay, B, Asp, Bd) if orient == 0 else orc.dds(lay, B, Ad, Asp)
            res[name] = bool(np.array_equal(sum(pieces), full)) and all(np.any(p) for p in pieces)
    if rank == 0:
        out.update(res)
    dist.destroy_process_group()


def test_two_ranks_split_dsd_and_dds_gloo():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_spmm_split_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out["dsd"] and out["dds"]   # disjoint rows / columns: the pieces add up to the whole, bit for bit
