"""The multi-GPU path is replicas only: the host logic that combines the ranks'
timings runs here on CPU as two gloo ranks (no GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_block_ingest_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
        slow = replicas.slowest_ms(ms, dist, "cpu")
        out[rank] = (slow, replicas.job_throughput(world, 200, slow))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slow, thr = res[r]
        assert slow == 15.0
        assert thr == pytest.approx(2 * 200 / 15e-3)


def test_single_rank_is_the_identity():
    assert replicas.slowest_ms(12.5) == 12.5
    assert replicas.job_throughput(1, 200, 100.0) == pytest.approx(2000.0)
