"""bench.py's multi-process path on CPU: two gloo ranks, a barrier, and the
max-over-ranks timing reduction (replicas only; the layer itself needs no
collective)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(10.0 + rank * 5.0, w)
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == 15.0 and out[1] == 15.0
