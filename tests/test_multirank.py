"""Rank plumbing of bench.py for N > 1 (independent replicas, no data-path
collective): two gloo ranks on the CPU run the same init / barrier /
max-over-ranks code torchrun drives on GPUs."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    w, r, local = bench.dist_init()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each replica reports its own step time; the job's time is the slowest
    t = bench.max_over_ranks(1.5 + rank, w)
    out[rank] = t
    # the reference arm runs on rank 0 only: other ranks return at once
    class A:
        workload = "causal_b1_h2_s128_d64"
        steps, warmup, ref_seconds = 1, 0, 0.1
    if rank != 0:
        assert bench.run_reference(A(), w, rank) is None
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    if torch.cuda.is_available():
        pytest.skip("checks the CPU (gloo) path")
    world = 2
    port = _free_port()
    # spawn, not fork: the process may already run OpenMP threads (the oracle)
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 2.5
