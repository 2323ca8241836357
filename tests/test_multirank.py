"""The N-GPU benchmark runs independent replicas (one batch per rank, no data-path
collective); only the step time is reduced across ranks (max) for the whole-job number.
Checked here with two gloo ranks on the CPU.  Also the pages' expert parallelism across
processes ("Serving Solar Open 2 (NVFP4) on DGX Spark", section on expert parallelism in
b12x: contiguous expert shards, each rank's output the partial sum of its local experts,
added by an all-reduce): two gloo ranks each run the oracle on one half of the experts and
the all-reduced partials equal the full layer."""
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


def _shard_rank_main(rank, world, port, out):
    import numpy as np
    import torch

    import oracle
    import synth
    from helpers import build_layer, slice_layer
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = synth.CONFIGS["tiny"]
        T, H, I, E, k = c["T"], c["H"], c["I"], c["E"], c["k"]
        layer = build_layer(0, H, I, E)
        wr = synth.router_weight(0, E, H)
        x = synth.activations(0, T, H)
        per = E // world
        lo = rank * per
        # contiguous shard [lo, lo + per); exactly one rank adds the shared expert
        cfg = oracle.make_cfg(T, H, I, E, k, E_loc=per, off=lo, add_shared=int(rank == 0),
                              inter_gs=1024.0)
        part = oracle.moe_forward(cfg, x, slice_layer(layer, lo, lo + per), router_w=wr)
        t = torch.from_numpy(np.ascontiguousarray(part.out))
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        if rank == 0:
            full = oracle.moe_forward(oracle.make_cfg(T, H, I, E, k, inter_gs=1024.0), x, layer,
                                      router_w=wr)
            out["err"] = float(np.max(np.abs(t.numpy() - full.out)))
            out["scale"] = float(np.max(np.abs(full.out)))
            out["pairs"] = int(len(part.pairs))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_all_reduce_oracle_shard_partials_to_the_full_layer():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert 0 < res["pairs"] < 16 * 2
    assert res["err"] <= 1e-12 * res["scale"], res
