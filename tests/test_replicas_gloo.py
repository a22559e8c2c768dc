"""The multi-GPU form of the benchmark is replicas only (the search does not
shard): each rank takes its own slice of the sources and the timing is the
maximum over ranks, the edge count the sum. This checks that host logic with
two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    sources = list(range(100, 116))
    mine = bench.rank_sources(sources, r, ws)
    t_max = bench.max_over_ranks(torch, ws, 1.0 + r, "cpu")
    e_sum = bench.sum_over_ranks(torch, ws, float(len(mine)), "cpu")
    bench.barrier(torch, ws)
    out[rank] = (ws, r, mine, t_max, e_sum)
    dist.destroy_process_group()


def test_two_rank_replica_split_and_reductions():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    r0, r1 = out[0], out[1]
    assert r0[0] == r1[0] == 2
    assert sorted(r0[2] + r1[2]) == list(range(100, 116))
    assert not set(r0[2]) & set(r1[2])
    assert r0[3] == r1[3] == 2.0          # max of (1.0, 2.0)
    assert r0[4] == r1[4] == 16.0         # all sources counted once


def test_rank_sources_with_fewer_sources_than_ranks():
    import bench
    assert bench.rank_sources([7], 3, 4) == [7]
    assert bench.rank_sources([1, 2, 3], 1, 2) == [2]
