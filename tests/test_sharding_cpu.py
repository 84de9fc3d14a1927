"""Multi-rank host logic on CPU (gloo, world size 2).

Rows are independent, so a batch is partitioned into contiguous row ranges
(row_range), one per rank: every rank selects its own rows and writes its
own slice of the outputs, and ranks exchange only the slowest time and the
total row count for the benchmark line.  These tests check that the ranges
cover every row exactly once, that the ranks' slices (the oracle on each
rank's rows) join to the oracle's answer on the whole batch with two real
processes, and the time / row-count reduction.
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


def _partition_worker(rank, world, port, out):
    """Every rank selects its row range of one batch (the oracle stands in
    for the GPU call); the slices are gathered for the check only."""
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    import oracle
    import top_selection_deepselect_gb300 as ds
    import workloads
    bits, _ = workloads.generate(7, 300, "bf16", "levels", seed=11)
    row_len = np.array([300, 17, 0, 250, 9, 300, 64], dtype=np.int32)
    r0, r1 = ds.row_range(rank, world, bits.shape[0])
    idx, val = oracle.topk(np.ascontiguousarray(bits[r0:r1]), "bf16", 20, row_len=row_len[r0:r1])
    parts = [None] * world
    dist.all_gather_object(parts, (r0, r1, idx.tolist(), val.tolist()))
    if rank == 0:
        ref_idx, ref_val = oracle.topk(bits, "bf16", 20, row_len=row_len)
        parts.sort()
        out["cover"] = [(a, b) for a, b, _, _ in parts]
        out["idx_equal"] = bool(np.array_equal(np.concatenate([np.array(p[2], np.int32).reshape(-1, 20)
                                                                for p in parts]), ref_idx))
        out["val_equal"] = bool(np.array_equal(np.concatenate([np.array(p[3], np.uint16).reshape(-1, 20)
                                                                for p in parts]), ref_val))
    dist.barrier()
    dist.destroy_process_group()


def test_row_ranges_cover_every_row_once():
    sys.path.insert(0, ROOT)
    import top_selection_deepselect_gb300 as ds
    for rows in range(0, 41):
        for world in range(1, 10):
            ranges = [ds.row_range(r, world, rows) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == rows
            assert all(ranges[i][1] == ranges[i + 1][0] for i in range(world - 1))
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0


def test_bench_rank_rows_weak_and_strong():
    sys.path.insert(0, ROOT)
    import bench
    # weak: every rank gets `rows` rows of a batch of rows * world
    assert [bench.rank_rows(r, 4, 256, "weak") for r in range(4)] == \
        [(0, 256, 1024), (256, 512, 1024), (512, 768, 1024), (768, 1024, 1024)]
    # strong: the workload's rows split across the ranks
    assert [bench.rank_rows(r, 3, 32, "strong")[:2] for r in range(3)] == [(0, 11), (11, 22), (22, 32)]


def test_rank_slices_join_to_the_whole_answer_two_processes():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_partition_worker, args=(world, port, out), nprocs=world,
                           start_method="spawn")
        res = dict(out)
    assert res["cover"] == [(0, 4), (4, 7)]
    assert res["idx_equal"] and res["val_equal"]


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
