"""bench.py's multi-rank path on CPU: two gloo ranks, each a replica of the
workload; the job value is the tokens of all ranks over the slowest rank's
time (replicas only: no collective on the data path)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r) == (world, rank)
    elapsed = [100.0, 250.0][rank]  # ms; rank 1 is the slow one
    value, worst = bench.aggregate_throughput(8192, 10, elapsed, w, torch.device("cpu"))
    out[rank] = (value, worst)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_rank_aggregation_uses_slowest_rank():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        value, worst = out[rank]
        assert worst == 250.0
        assert value == pytest.approx(2 * 8192 * 10 / 0.250)


def test_single_rank_is_identity():
    import bench
    v, worst = bench.aggregate_throughput(100, 4, 50.0, 1, torch.device("cpu"))
    assert worst == 50.0 and v == pytest.approx(100 * 4 / 0.05)
