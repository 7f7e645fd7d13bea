"""Expert parallelism on CPU: world sizes 2 and 3 over gloo, each rank computing its partial sum with the oracle.

Checks the host side of int4_grouped_expert_router_gb300.ep: the expert ownership rule matches the oracle's,
the gather returns every rank's partial rows in rank order on every rank, and the rank-order sum reproduces
the oracle's expert-parallel block bit for bit (and the one-rank block up to rounding) on every rank.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.moe as O
from int4_grouped_expert_router_gb300 import ep, synth

D, I, E, K, S = 16, 8, 9, 3, 3


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    experts = {}
    for e in range(E):
        trip = []
        for which, (r, c, gs) in zip("gud", ((I, D, 0), (I, D, 4), (D, I, 2))):
            p, sc = synth.expert_tensor(synth.stream_seed(300, e, which), r, c, gs)
            trip.append(O.Tensor(p, sc, r, c, gs))
        experts[e] = tuple(trip)
    x = synth.normal(synth.stream_seed(301, "x"), S * D).reshape(S, D)
    resid = synth.normal(synth.stream_seed(301, "r"), S * D).reshape(S, D)
    Wr = synth.normal(synth.stream_seed(301, "Wr"), E * D).reshape(E, D) * 0.1
    idx, w, n, _ = O.router_select(x, Wr, None, K, 0.0, True, 2.5)
    return experts, x, resid, idx, w, n


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        experts, x, resid, idx, w, n = _problem()
        mine = {e: t for e, t in experts.items() if ep.owner(e, world) == rank}  # this rank's table
        si, sw, sn = O.shard_routes(idx, w, n, rank, world)
        partial = O.expert_group(x, mine, si, sw, sn, None)
        parts = ep.gather_partials(torch.from_numpy(partial), None)
        acc = parts[0].numpy()
        for r in range(1, world):
            acc = acc + parts[r].numpy()
        out[rank] = (resid + acc, parts.numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world):
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        return dict(out)


def test_owner_matches_oracle():
    for world in (1, 2, 3, 8):
        assert [ep.owner(e, world) for e in range(40)] == [O.expert_owner(e, world) for e in range(40)]


def test_expert_parallel_reduce_over_gloo():
    experts, x, resid, idx, w, n = _problem()
    ref1 = O.expert_group(x, experts, idx, w, n, resid)
    for world in (2, 3):
        res = _run(world)
        want = O.ep_layer(x, experts, idx, w, n, world, resid)
        y0, parts0 = res[0]
        for r in range(world):
            y, parts = res[r]
            assert np.array_equal(parts, parts0), (world, r)  # the same stack, in rank order, everywhere
            assert np.array_equal(y, want), (world, r)
        for r in range(world):  # stack slot r holds rank r's own partial
            si, sw, sn = O.shard_routes(idx, w, n, r, world)
            assert np.array_equal(parts0[r], O.expert_group(x, experts, si, sw, sn, None)), (world, r)
        assert np.allclose(y0, ref1, rtol=1e-12, atol=1e-12)


class _OracleDevice:
    """Stand-ins for the library calls ExpertParallelLayer makes, computed by the oracle on CPU tensors."""

    def __init__(self, experts):
        self.experts, self.pending = experts, None

    def coli_router_select(self, ctx, x, Wr, bias, K, topp, norm_topk, routed_scale, idx, w, n_sel):
        i, ww, n, _ = O.router_select(x.numpy(), Wr.numpy(), None if bias is None else bias.numpy(), K, topp,
                                      norm_topk, routed_scale)
        idx.copy_(torch.from_numpy(i))
        w.copy_(torch.from_numpy(ww))
        n_sel.copy_(torch.from_numpy(n))

    def coli_routes_shard(self, ctx, idx, w, n_sel, rank, world, idx_out, w_out, n_out):
        i, ww, n = O.shard_routes(idx.numpy(), w.numpy(), n_sel.numpy(), rank, world)
        idx_out.copy_(torch.from_numpy(i))
        w_out.copy_(torch.from_numpy(ww))
        n_out.copy_(torch.from_numpy(n))

    def coli_expert_group_issue(self, ctx, x, idx, w, n_sel, K):
        assert self.pending is None
        self.pending = (x.numpy(), idx.numpy(), w.numpy(), n_sel.numpy())
        return 0

    def coli_expert_group_take(self, ctx, resid, y):
        x, idx, w, n = self.pending
        self.pending = None
        p = O.expert_group(x, self.experts, idx, w, n, None)
        y.copy_(torch.from_numpy(p if resid is None else resid.numpy() + p))

    def coli_partials_reduce(self, ctx, parts, resid, y):
        acc = parts[0].numpy().astype(np.float64)
        for r in range(1, parts.shape[0]):
            acc = acc + parts[r].numpy()
        y.copy_(torch.from_numpy(acc if resid is None else resid.numpy() + acc))


def _layer_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        experts, x, resid, _, _, _ = _problem()
        Wr = synth.normal(synth.stream_seed(301, "Wr"), E * D).reshape(E, D) * 0.1
        mine = {e: t for e, t in experts.items() if ep.owner(e, world) == rank}
        ep.B = _OracleDevice(mine)  # this process only: the layer's library calls go to the oracle
        layer = ep.ExpertParallelLayer(None, rank, world)
        y = torch.empty(S, D, dtype=torch.float64)
        idx, w, n = layer.step(torch.from_numpy(x), torch.from_numpy(Wr), None, K, 0.0, True, 2.5,
                               torch.from_numpy(resid.astype(np.float64)), y)
        out[rank] = (y.numpy(), idx.numpy(), w.numpy(), n.numpy())
        try:
            layer.step(torch.from_numpy(x).to(torch.bfloat16), torch.from_numpy(Wr), None, K, 0.0, True, 2.5, None, y)
            out[f"bf16-{rank}"] = "accepted"
        except ValueError:
            out[f"bf16-{rank}"] = "rejected"
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_expert_parallel_layer_over_gloo():
    """ExpertParallelLayer's call order (route, shard, issue, take, gather, reduce) with world size 2, the
    library calls computed by the oracle: every rank ends with the oracle's expert-parallel block."""
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_layer_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    experts, x, resid, idx, w, n = _problem()
    want = O.ep_layer(x, experts, idx, w, n, world, resid)
    for r in range(world):
        y, i, ww, nn = res[r]
        assert np.array_equal(i, idx) and np.array_equal(nn, n)
        assert np.allclose(y, want, rtol=1e-6, atol=1e-6)  # the exchanged partial rows are f32
        assert res[f"bf16-{r}"] == "rejected"
