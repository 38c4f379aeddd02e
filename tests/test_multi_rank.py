"""The N > 1 benchmark path on CPU: two gloo ranks, max-over-ranks step time and
summed work (the bench's weak-scaling aggregation; no data-path collective)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms, work = bench.aggregate(10.0 + 5.0 * rank, 100.0 * (rank + 1), world)
    assert bench.dist_env() == (world, rank, rank)
    q.put((rank, ms, work))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_aggregation(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for _, ms, work in got:
        assert ms == 15.0          # max over ranks
        assert work == 300.0       # sum over ranks


def test_single_rank_identity():
    import bench

    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)
