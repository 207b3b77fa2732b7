"""The bench's multi-rank timing path on CPU: two gloo ranks, barrier, and the
max-over-ranks reduction that turns per-replica times into the job time."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench

    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    t = bench.max_over_ranks(dist, 1.5 + rank, device="cpu")
    out[rank] = t
    dist.destroy_process_group()


def test_two_rank_max_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.0) == 3.0
