"""Host logic of bench.py's N > 1 path (independent replicas, max-over-ranks timing) on a
world-size-2 gloo group on the CPU.  No GPU."""
from __future__ import annotations

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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [0.25, 0.40][rank]
    t = bench.max_over_ranks(local, dist, torch.device("cpu"))
    rate = bench.whole_job_rate(1000.0, world, t)
    out[rank] = (t, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_is_max_and_rate_counts_both_replicas():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    t, rate = out[0]
    assert t == 0.40
    assert abs(rate - 2 * 1000.0 / 0.40) < 1e-9


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(0.3) == 0.3
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
