"""The benchmark's multi-rank path (independent replicas, no data exchange):
two gloo ranks on CPU check the max-over-ranks timing and the whole-job value."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r "took" 10 + 5 r milliseconds
    slowest = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)
    value = bench.job_throughput(1e12, world, 4, slowest)
    dist.barrier()
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_over_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 4 steps x 1 TFLOP in 15 ms
    assert abs(res[0][1] - 2 * 4 / 0.015) < 1e-6
    assert res[0][1] == res[1][1]


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert abs(bench.job_throughput(2e12, 1, 10, 20.0) - 1000.0) < 1e-9
