"""The replicas path of bench.py (N > 1): ranks reduce their timed region to
the slowest rank's time and the sum of their bytes.  world_size 2 over gloo
on the CPU."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 12.5][rank]
    nbytes = [1e9, 3e9][rank]
    q.put((rank, bench.reduce_over_ranks(ms, nbytes, "cpu"), bench.dist_info()))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_reduce_max_time_and_total_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (ms, nbytes), (ws, rk, local) in out:
        assert ms == 12.5 and nbytes == 4e9
        assert ws == 2 and rk == rank


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.0, 7.0) == (3.0, 7.0)
