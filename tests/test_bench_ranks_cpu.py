"""The multi-GPU timing path of bench.py on CPU: two gloo ranks, each with
its own batch (weak scaling, no data-path collective); the job's time is the
slowest rank's and its throughput counts every rank's tokens."""
import os
import socket

import pytest
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
    ms = [120.0, 150.0][rank]          # per-rank device time of 100 steps
    e2e = [0.20, 0.17][rank]           # per-rank end-to-end seconds
    dist.barrier()
    ms_max, e2e_max = bench.combine_ranks(ms, e2e, world, "cpu")
    v = bench.weak_scaling_value(world, 64, 100, ms_max / 1e3)
    out[rank] = (ms_max, e2e_max, v)
    dist.destroy_process_group()


def test_two_rank_timing_takes_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms_max, e2e_max, v = out[r]
        assert ms_max == 150.0 and e2e_max == 0.20
        assert v == pytest.approx(2 * 64 * 100 / 0.150)


def test_single_rank_is_identity():
    import bench
    assert bench.combine_ranks(12.5, 0.3, 1, "cpu") == (12.5, 0.3)
    assert bench.weak_scaling_value(1, 64, 10, 0.5) == pytest.approx(1280.0)
