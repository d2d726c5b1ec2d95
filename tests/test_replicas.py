"""The N>1 path of bench.py runs independent replicas (the step has no
cross-request exchange).  Its host logic -- the maximum of the per-rank step
times and the whole-job rate -- is checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        assert (r, w) == (rank, world)
        total_ms = 100.0 + 50.0 * rank          # rank 1 is the slower replica
        m = bench.reduce_max(total_ms, world, "cpu")
        bench.barrier(world)
        out[rank] = (m, bench.whole_job_rate(1000, world, m))
    finally:
        dist.destroy_process_group()


def test_two_rank_replica_reduction():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1]
    m, rate = out[0]
    assert m == 150.0
    assert rate == pytest.approx(2 * 1000 / 0.150)


def test_single_rank_reduction_is_identity():
    assert bench.reduce_max(12.5, 1) == 12.5
    assert bench.whole_job_rate(10, 1, 2000.0) == pytest.approx(5.0)
