"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1
(replicas only: the path has no data exchange, the only collectives are the
timing barrier and the max/sum of per-rank numbers)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_setup()
    dev = torch.device("cpu")
    bench.barrier(w)
    mx = bench.max_over_ranks(1.5 + r, w, dev)
    sm = bench.sum_over_ranks(10.0 * (r + 1), w, dev)
    q.put((r, w, local, mx, sm))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for r, (rank, w, local, mx, sm) in enumerate(got):
        assert (rank, w, local) == (r, world, r)
        assert mx == 2.5 and sm == 30.0


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    assert bench.sum_over_ranks(3.0, 1, None) == 3.0
