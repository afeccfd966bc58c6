"""The N>1 host path of bench.py on CPU: two gloo ranks (no GPU).

Requests are independent, so the path shards by request with no collective
in the data path; the only cross-rank operations are the timing barrier and
the max-over-ranks reduction of the elapsed time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    mx = bench.max_over_ranks(ms, dist, "cpu")
    shard = list(bench.rank_requests(7, world, rank))
    dist.barrier()
    q.put((rank, mx, shard, bench.aggregate_blocks_per_s(world, 3, 4, mx)))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_disjoint_shards():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]                 # both ranks report the slowest
    shards = [r[2] for r in res]
    assert sorted(shards[0] + shards[1]) == list(range(7))     # every request exactly once
    assert not set(shards[0]) & set(shards[1])
    assert res[0][3] == pytest.approx(2 * 3 * 4 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(12.5) == 12.5
    assert list(bench.rank_requests(5, 1, 0)) == list(range(5))
