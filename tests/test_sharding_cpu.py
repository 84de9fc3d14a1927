"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

Rows are independent, so every rank runs its own batch and ranks exchange
only the slowest time and the total row count; this checks that reduction
with two real processes.
"""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, rows = bench.reduce_over_ranks(10.0 + 5.0 * rank, 64 * (rank + 1), dist)
    out[rank] = (ms, rows)
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_over_ranks_two_processes():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:  # no fork of this multi-threaded process
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == (15.0, 64 + 128)


def test_reduce_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, 7, None) == (3.5, 7)
