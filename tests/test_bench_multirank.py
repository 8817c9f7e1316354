"""The benchmark's multi-rank bookkeeping (replicas, max over ranks) on two
gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank 1 is the slow one on the first timing, rank 0 on the second
    local = [10.0 + 5.0 * rank, 30.0 - 4.0 * rank, 1.0 + rank]
    got = bench.max_over_ranks(local, world, torch.device("cpu"))
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == [15.0, 30.0, 2.0]


def test_aggregate_is_all_ranks_work_over_slowest_time():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 100 steps x 1e12 FLOP in 200 ms (the slower rank) -> 1000 TFLOPS
    assert bench.aggregate_tflops(1e12, 100, 200.0, 2) == pytest.approx(1000.0)
    assert bench.aggregate_tflops(1e12, 100, 200.0, 1) == pytest.approx(500.0)
