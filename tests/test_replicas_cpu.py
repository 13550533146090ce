"""Multi-rank host logic of the bench (replicas only): two gloo ranks on the CPU.

Each rank runs an independent replica; the job time is the slowest rank's
time and the job throughput counts every rank's rows."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as td
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    td.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r measured (2 + r) ms per step and (3 + 2r) ms end to end
    ms, e2e = bench.reduce_over_ranks([2.0 + rank, 3.0 + 2 * rank], world, "cpu")
    out[rank] = (ms, e2e, bench.job_rows_per_s(48, world, ms))
    td.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, e2e, value = res[r]
        assert ms == 3.0 and e2e == 5.0
        assert value == pytest.approx(48 * 2 / 3e-3)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.job_rows_per_s(4, 1, 2.0) == pytest.approx(2000.0)
