"""The multi-rank arithmetic of bench.py on CPU: two gloo ranks, each with
its own elapsed time, agree on the maximum and on the whole-job value."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        elapsed = [12.5, 20.0][rank]           # the second rank is slower
        bench.barrier()
        m = bench.reduce_max(elapsed, "cpu")
        v = bench.job_throughput(4096, 10, world, m)
        out[rank] = (m, v)
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    m, v = out[0]
    assert m == 20.0
    assert v == pytest.approx(2 * 4096 * 10 / 0.020)


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.job_throughput(100, 2, 1, 1000.0) == pytest.approx(200.0)
