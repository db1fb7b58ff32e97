"""The N-GPU host logic of bench.py, run as 2 gloo ranks on the CPU.

Each GPU runs an independent replica of the workload (requests are
independent, so the path shards with no data exchange).  What crosses ranks
is only the timing: the job takes as long as its slowest replica, and the
whole-job throughput counts every replica's bytes.
"""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # replica times differ; every rank must see the slowest one
        slowest = bench.reduce_max(10.0 + 5.0 * rank, dist, "cpu")
        value = bench.whole_job_gbs(2e9, 100, world, slowest)
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_whole_job_value():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0] == out[1]
    slowest, value = out[0]
    assert slowest == 15.0
    assert value == pytest.approx(2 * 2e9 * 100 / 15.0 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(3.5, None, "cpu") == 3.5
    assert bench.whole_job_gbs(1e9, 10, 1, 2.0) == pytest.approx(5.0)
