"""The multi-process host logic of bench.py on CPU: two gloo ranks, each with
its own timing, agree on the slowest rank's time and the whole-job value.
(On GPUs the same functions run over NCCL; nothing on the data path is
exchanged between ranks.)"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 17.0][rank]
        total = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        out[rank] = (total, bench.whole_job_tflops(world, 2.0e12, 10, total))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == out[1]
    total, value = out[0]
    assert total == 17.0
    assert value == pytest.approx(2 * 2.0e12 * 10 / 17.0e-3 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.0, None, torch.device("cpu")) == 3.0
    assert bench.whole_job_tflops(1, 1.0e12, 1, 1.0) == pytest.approx(1000.0)
