"""The benchmark's multi-rank path on CPU (gloo, world size 2): replicas share no data;
the only collectives are the barrier and the max-over-ranks of the timed region."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    import torch.distributed as dist
    r, w, lr = bench.dist_init()
    assert (r, w, lr) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier()
    # Each replica reports its own elapsed time; every rank gets the slowest one.
    got = bench.max_over_ranks(10.0 + rank)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert res == [(0, 11.0), (1, 11.0)]


def test_single_rank_is_identity(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    assert bench.dist_init() == (0, 1, 0)
    assert bench.max_over_ranks(3.5) == 3.5
    bench.barrier()
