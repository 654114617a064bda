"""The multi-GPU path of the benchmark is replicas only (the (batch, head) slices never
exchange data): its host logic -- max of the ranks' step times, whole-job throughput from
all ranks' FLOPs -- runs here as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]                      # rank 1 is the slower replica
        m = bench.max_over_ranks(ms, world)
        out[rank] = (m, bench.job_tflops(1e12, world, m))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        m, tf = res[rank]
        assert m == 5.0
        assert tf == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_tflops(2e12, 1, 4.0) == pytest.approx(500.0)
