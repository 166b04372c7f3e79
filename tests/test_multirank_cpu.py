"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

The linear shards with no exchange step, so N GPUs run independent replicas;
the only cross-rank work is taking the slowest rank's time and scaling the
job throughput by the rank count.  Run here as world_size 2 over gloo."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench  # noqa: E402  (repo root is on sys.path via conftest)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = [3.0, 5.0][rank]
        slowest = bench.max_over_ranks(ms, ws, torch.device("cpu"))
        value = bench.job_throughput(1e9, slowest, ws)
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    ws = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
    assert out[0] == out[1]
    slowest, value = out[0]
    assert slowest == 5.0
    # 2 ranks x 1 GB in 5 ms = 400 GB/s for the job
    assert value == pytest.approx(400.0)


def test_single_rank_passthrough():
    assert bench.max_over_ranks(2.5, 1, torch.device("cpu")) == 2.5
    assert bench.job_throughput(1e9, 1.0, 1) == pytest.approx(1000.0)
