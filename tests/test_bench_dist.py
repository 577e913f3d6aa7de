"""bench.py's multi-rank timing helpers on CPU ranks (gloo, world size 2)."""
import os
import socket
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    out[rank] = bench.max_over_ranks(1.5 + rank, world)   # each rank reports its own time
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn",
                       join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}
