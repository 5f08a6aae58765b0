"""Host logic of bench.py for N > 1 ranks (CPU, gloo, world size 2).

The decode path shards by request with no data-path collective: each rank runs
its own replica and the only cross-rank operations are a barrier and the
reduction of timing scalars (slowest rank's time, total units)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist = bench.dist_init(world, "gloo")
    bench.barrier(dist)
    ms, units = bench.aggregate(dist, 10.0 + 5.0 * rank, 1000.0 * (rank + 1))
    results[rank] = (ms, units)
    # the reference arm runs on rank 0 only; other ranks return without work
    if rank != 0:
        results[10 + rank] = bench.run_reference(bench.parse_args(["--impl", "reference"]))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_rank_aggregation_uses_slowest_rank_and_total_units():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        ms, units = res[rank]
        assert ms == pytest.approx(15.0)        # max over ranks
        assert units == pytest.approx(3000.0)   # sum over ranks
    assert res[11] is None


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(None, 12.5, 7.0) == (12.5, 7.0)
    assert bench.dist_init(1, "gloo") is None
