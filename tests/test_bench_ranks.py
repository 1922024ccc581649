"""bench.py's multi-rank logic on CPU: world_size-2 gloo ranks barrier,
take the max of their timed spans and sum the units they processed (weak
scaling: each rank owns an independent batch, no data-path collective)."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    t = bench.reduce_max(1.0 + rank, w)       # rank 1 was slower
    units = bench.reduce_sum(100.0 * (rank + 1), w)
    q.put((rank, t, units))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_sum_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, units in got:
        assert t == 2.0 and units == 300.0


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.reduce_sum(7.0, 1) == 7.0
