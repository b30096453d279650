"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing
its own replica, agree on the slowest rank's time (the reported step time)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, _ = bench.dist_env()
    assert (ws, r) == (world, rank)
    mine = 1.5 + rank * 2.25           # each replica's own time
    out[rank] = bench.max_over_ranks(mine)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    assert out[0] == out[1] == pytest.approx(3.75)


def test_max_over_ranks_without_a_group_is_identity():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
