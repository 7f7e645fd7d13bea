"""The multi-rank (replicas) logic of bench.py on CPU: world size 2 over gloo.

Each rank times its own tokens; the job time is the slowest rank's, and the per-layer figure
divides it by the layers all ranks ran. The reference arm prints only on rank 0.
"""
import contextlib
import io
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(local_ms[rank], dist, "cpu")
        out[rank] = (m, bench.job_us_per_layer(m, 10, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_world2_job_time_is_slowest_rank():
    world, port = 2, _free_port()
    local_ms = [1.25, 3.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, local_ms, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        m, us = res[r]
        assert m == max(local_ms)
        assert us == pytest.approx(max(local_ms) * 1000.0 / (10 * world))


def test_single_rank_is_identity():
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.job_us_per_layer(2.5, 10, 1) == pytest.approx(250.0)


def test_ranks_get_distinct_tokens():
    seeds = {bench.token_seed(r, s) for r in range(8) for s in range(1000)}
    assert len(seeds) == 8 * 1000


def test_reference_arm_prints_on_rank0_only():
    class A:
        workload = "decode"
        steps = 1
        warmup = 0
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.reference_arm(A(), 1, 2) == 0
    assert buf.getvalue() == ""


def _ep_rank_main(rank, world, port, local_ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        owned = [e for e in range(256) if bench.ep_owned(e, rank, world)]
        seeds = [bench.ep_token_seed(s) for s in range(20)]
        m = bench.max_over_ranks(local_ms[rank], dist, "cpu")
        out[rank] = (owned, seeds, m, bench.ep_job_us_per_layer(m, 10))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_ranks_split_experts_and_share_tokens(world):
    """--gpus N with expert parallelism: the ranks own disjoint experts that cover the layer, route the same
    tokens, and the job's per-layer time is the slowest rank's time divided by the layers (not by N: the ranks
    run each layer together)."""
    port = _free_port()
    local_ms = [1.0 + r for r in range(world)]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_ep_rank_main, args=(world, port, local_ms, out), nprocs=world, join=True)
        res = dict(out)
    owned = [set(res[r][0]) for r in range(world)]
    assert set().union(*owned) == set(range(256))
    assert sum(len(o) for o in owned) == 256
    assert all(res[r][1] == res[0][1] for r in range(world))
    for r in range(world):
        assert res[r][2] == max(local_ms)
        assert res[r][3] == pytest.approx(max(local_ms) * 1000.0 / 10)
