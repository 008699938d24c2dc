"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2).

The layer shards without any exchange (directions and batch rows are
independent), so a multi-GPU run is N independent replicas: the only
cross-rank work is the barrier around the timed region and the max / sum
reductions of the timings and FLOP counts, which these tests cover.  The
reference arm under torchrun must print on rank 0 only and let the other
ranks exit without work.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    mx = bench.max_over_ranks(1.5 + rank, world)
    sm = bench.sum_over_ranks(10.0 * (rank + 1), world)
    r, w, l = bench.dist_env()
    q.put((rank, mx, sm, r, w, l))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, sm, r, w, l in res:
        assert mx == 2.5 and sm == 30.0 and r == rank and w == 2 and l == rank


def test_single_rank_reductions_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.sum_over_ranks(7.0, 1) == 7.0


def test_reference_arm_nonzero_rank_exits_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
