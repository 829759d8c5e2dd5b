"""The multi-rank path of bench.py on CPU: two gloo ranks (127.0.0.1) time
different amounts, and both see the slowest rank's time; the whole-job value
counts every rank's work over that time (replicas, weak scaling)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [2.0, 3.5][rank]
    ms = bench.max_over_ranks(local_ms, world, dist, "cpu")
    dist.barrier()
    out[rank] = (ms, bench.job_tflops(world, 161.06e9, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 3.5
    assert out[0][1] == pytest.approx(2 * 161.06e9 / 3.5e-3 / 1e12)


def test_one_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(1.25, 1, None, "cpu") == 1.25
    assert bench.job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
