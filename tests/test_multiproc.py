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


def test_reference_arm_under_torchrun_prints_one_line():
    """bench.py --impl reference launched as the driver launches N > 1 (torchrun, two gloo ranks on
    CPU): rank 0 alone times the oracle and prints one JSON line; the other rank exits 0.  The
    small config-1 workload keeps the oracle's inputs quick to draw on the CPU."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--config", "1", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
