"""The multi-GPU path is N independent replicas (the (sequence, head) units
need no exchange).  What the ranks share is the timing: the job's time is the
slowest rank's and the job's throughput counts every rank's tokens.  Tested
here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, outdir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        # rank 1 is the slow one: 30 ms over 3 steps
        ms, value = bench.replica_throughput(15.0 if rank == 0 else 30.0, 3, 1000, dist, "cpu")
        with open(os.path.join(outdir, "rank%d" % rank), "w") as f:
            f.write("%r %r" % (ms, value))
    finally:
        dist.destroy_process_group()


def test_replica_timing_is_max_over_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank, args=(port, str(tmp_path)), nprocs=2, join=True)
    for rank in (0, 1):
        ms, value = map(float, open(tmp_path / ("rank%d" % rank)).read().split())
        assert ms == pytest.approx(10.0)
        assert value == pytest.approx(2 * 1000 / 10e-3)


def test_single_process_throughput():
    ms, value = bench.replica_throughput(20.0, 4, 500)
    assert ms == pytest.approx(5.0) and value == pytest.approx(500 / 5e-3)
