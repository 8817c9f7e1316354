"""The benchmark's bookkeeping on the CPU: multi-rank replicas (max over
ranks, two gloo ranks), byte accounting, and the source hash that keeps
recorded counters tied to the kernel they were taken on."""
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


def test_sparse_byte_accounting():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    K, N, E, R = 6144, 4096, 128, 2048
    dense, sparse = bench.gemm_bytes(K, N, E, R, R), bench.sparse_gemm_bytes(K, N, E, R, R)
    io = bench.gemm_bytes(K, N, 0, R, R)
    assert io == bench.sparse_gemm_bytes(K, N, 0, R, R)
    # weights: 0.375 B per element sparse (kept codes, indices, scales), 0.5625 dense
    assert (sparse - io) * 0.5625 == pytest.approx((dense - io) * 0.375)
    assert bench.step_bytes(E, sparse=True) < bench.step_bytes(E)


def test_source_hash_ignores_comments_only():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) {\n  return x + 1;  // one\n}\n"
    b = "/* doc */ int f(int x) {\n\n  return x + 1;\n}  // trailing\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.normalised_source(a) == bench.normalised_source(b)
    assert bench.normalised_source(a) != bench.normalised_source(c)
    assert bench.kernel_source_hash() == bench.kernel_source_hash()
