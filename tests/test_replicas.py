"""The multi-GPU path is replicas only: each rank runs the whole workload on its own GPU and the
timing is the maximum over ranks.  These tests run that host logic as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [10.0 + rank, 3.0 - rank, 1.5 * (rank + 1)]
        got = bench.max_over_ranks(times, world)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    want = [11.0, 3.0, 3.0]
    assert out[0] == want and out[1] == want


def test_single_rank_is_identity():
    assert bench.max_over_ranks([1.0, 2.5], 1) == [1.0, 2.5]


def test_replica_throughput_counts_all_ranks():
    # two replicas of 1e12 flop each, the slower one taking 10 ms: 2e12 / 0.01 s = 200 TFLOP/s
    assert bench.replica_throughput(1e12, 10.0, 2) == pytest.approx(200.0)
    assert bench.replica_throughput(1e12, 10.0, 1) == pytest.approx(100.0)
