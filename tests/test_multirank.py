"""The benchmark's multi-rank plumbing on CPU (gloo, two ranks): each rank is an
independent replica; the step time is the maximum over ranks; only rank 0 runs the
reference (oracle) arm and prints."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    r, w, lr = bench.dist_info()
    assert (r, w, lr) == (rank, world, rank)
    t = bench.max_over_ranks(1.0 + rank, world)
    bench.barrier(world)
    args = type("A", (), dict(workload="tiny", T=8, experts=None, routing=None, capacity=None, steps=1, warmup=0))()
    ref, _ = bench.run_reference(args, rank, world, rank) if rank != 0 else (None, None)
    out[rank] = (t, ref is None)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == 2.0 and res[1][0] == 2.0
    assert res[1][1]  # a non-zero rank does no reference work
