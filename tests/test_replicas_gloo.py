"""The multi-GPU path of the benchmark is replicas only (each rank runs its own chunk; the only
collectives are the timing barrier and a max over ranks).  This covers that host logic with two
gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [2.5, 3.75][rank]                 # the second rank is the slow one
        dist.barrier()
        slowest = bench.max_over_ranks(local_ms, world)
        rate = bench.replicas_rate(4096, world, slowest)
        # the reference arm: only rank 0 works and prints, the others return 0 at once
        rc = bench.run_reference(None, None, rank, world) if rank != 0 else 0
        results[rank] = (slowest, rate, rc)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    port = _free_port()
    results = mp.get_context("spawn").Manager().dict()   # no fork once CUDA may be initialised
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    for rank in range(world):
        slowest, rate, rc = results[rank]
        assert slowest == 3.75
        assert rate == pytest.approx(4096 * 2 / 3.75e-3)
        assert rc == 0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.replicas_rate(10, 1, 1.0) == pytest.approx(10000.0)
