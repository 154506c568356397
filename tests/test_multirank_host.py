"""bench.py's multi-rank host logic on CPU: two gloo ranks, each with its own
replica of the work (weak scaling), the slowest rank's time decides."""

import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 100.0 + 50.0 * rank  # rank 1 is slower
    m = bench.max_over_ranks(local_ms, world, device="cpu")
    v = bench.whole_job_value(2.0e12, 10, world, m)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        m, v = out[r]
        assert m == 150.0
        # 2 ranks x 2 TFLOP x 10 steps in 0.15 s
        assert abs(v - 2 * 2.0e12 * 10 / 0.150 / 1e12) < 1e-9


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.whole_job_value(1e12, 4, 1, 2.0) - 2000.0) < 1e-9
