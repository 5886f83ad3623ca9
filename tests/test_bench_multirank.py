"""The benchmark's multi-GPU path (independent replicas) on CPU: two gloo ranks agree on the
slowest rank's time and on the whole-job throughput.  No GPU needed."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.reduce_max(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        out[rank] = (ms, bench.job_throughput(1000, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == out[1]
    ms, tput = out[0]
    assert ms == 15.0
    assert tput == pytest.approx(2 * 1000 / 15e-3)


def test_single_process_is_identity():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.job_throughput(10, 1, 1.0) == pytest.approx(10000.0)
