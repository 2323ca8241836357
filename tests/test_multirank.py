"""The N-GPU benchmark runs independent replicas (one batch per rank, no data-path
collective); only the step time is reduced across ranks (max) for the whole-job number.
Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [0.42, 0.57][rank]  # each replica's own step time
        slowest = bench.max_over_ranks(ms, world, device="cpu")
        dist.barrier()
        out[rank] = (slowest, bench.job_tokens_per_s(world, 64, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slowest, tps = res[r]
        assert slowest == pytest.approx(0.57)
        assert tps == pytest.approx(2 * 64 / 0.57e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_tokens_per_s(1, 64, 0.5) == pytest.approx(128000.0)
