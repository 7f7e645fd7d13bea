"""Expert parallelism, the device steps on one GPU: ranks simulated one after another (no collective).

- coli_routes_shard against the oracle's shard_routes, slot for slot, for 2, 3 and 5 ranks (top-p rows included).
- Each simulated rank's partial sum (issue + take, no residual), stacked in rank order and reduced by
  coli_partials_reduce, against the oracle's expert-parallel block and against the one-GPU coli_expert_group.
- One rank through ExpertParallelLayer is bit-identical to coli_expert_group.
- A kept slot naming no expert sets COLI_E_ROUTE.
"""
import numpy as np
import pytest
import torch

import oracle.moe as O
from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.ep import ExpertParallelLayer
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import F32_RTOL, Ctx, assert_close, f32_atol, oracle_experts, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


CASES = [
    LayerConfig("ep-S1", D=512, I=256, E=16, K=8, routed_scale=2.5),
    LayerConfig("ep-S5-topp-g64", D=320, I=200, E=20, K=6, S=5, gs="mixed:64", topp=0.85),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_simulated_ranks_match_oracle(ctx, cfg):
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        r = layer.outputs()
        B.coli_router_select(ctx, xt, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale,
                             r["idx"], r["w"], r["n_sel"])
        y1 = torch.empty_like(xt)
        B.coli_expert_group(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K, rt, y1)
        idx, w, n = (to_np(r[k]) for k in ("idx", "w", "n_sel"))
        experts = oracle_experts(cfg, idx)
        for world in (2, 3, 5):
            parts = torch.empty(world, cfg.S, cfg.D, device="cuda")
            for rank in range(world):
                si, sw, sn = torch.empty_like(r["idx"]), torch.empty_like(r["w"]), torch.empty_like(r["n_sel"])
                B.coli_routes_shard(ctx, r["idx"], r["w"], r["n_sel"], rank, world, si, sw, sn)
                oi, ow, on = O.shard_routes(idx, w, n, rank, world)
                assert np.array_equal(to_np(si), oi) and np.array_equal(to_np(sw), ow) and np.array_equal(to_np(sn), on)
                B.coli_expert_group_issue(ctx, xt, si, sw, sn, cfg.K)
                B.coli_expert_group_take(ctx, None, parts[rank])
            y = torch.empty_like(xt)
            B.coli_partials_reduce(ctx, parts, rt, y)
            assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
            ref = O.ep_layer(to_np(xt), experts, idx, w, n, world, to_np(rt))
            print(cfg.name, world, assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), f"{cfg.name} world {world}"))
            assert_close(to_np(y), to_np(y1), F32_RTOL, f32_atol(ref), f"{cfg.name} world {world} vs one GPU")
    finally:
        layer.free()


def test_one_rank_layer_is_the_one_gpu_call(ctx):
    cfg = LayerConfig("ep-one", D=256, I=128, E=16, K=4, topp=0.9)
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        y = torch.empty_like(xt)
        idx, w, n = ExpertParallelLayer(ctx, 0, 1).step(xt, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk,
                                                         cfg.routed_scale, rt, y)
        y1 = torch.empty_like(xt)
        B.coli_expert_group(ctx, xt, idx, w, n, cfg.K, rt, y1)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        assert torch.equal(y, y1)
    finally:
        layer.free()


def test_unowned_kept_slot_is_reported(ctx):
    idx = torch.tensor([[3, -1, 5]], dtype=torch.int32, device="cuda")
    w = torch.tensor([[0.5, 0.25, 0.25]], device="cuda")
    n = torch.tensor([3], dtype=torch.int32, device="cuda")
    si, sw, sn = torch.empty_like(idx), torch.empty_like(w), torch.empty_like(n)
    B.coli_routes_shard(ctx, idx, w, n, 1, 2, si, sw, sn)
    assert B.coli_check_error(ctx) == B.COLI_E_ROUTE
    assert si.tolist() == [[3, 5, -1]] and sn.tolist() == [2]
    B.coli_routes_shard(ctx, idx, w, torch.tensor([1], dtype=torch.int32, device="cuda"), 1, 2, si, sw, sn)
    assert B.coli_check_error(ctx) == 0  # the bad slot is beyond n_sel: ignored
    assert si.tolist() == [[3, -1, -1]] and sn.tolist() == [1]


@pytest.mark.parametrize("world", [2, 3])
def test_each_rank_holds_only_its_experts(world):
    """The deployment shape of the expert-parallel bench: one context per simulated rank whose table holds only
    the experts e with e mod world == rank (DeviceLayer owned=...), every rank routing the same token itself;
    the rank-order reduce of their partials matches the oracle's expert-parallel block."""
    import bench
    cfg = LayerConfig("ep-owned", D=1024, I=256, E=16, K=8, routed_scale=2.5)
    ctxs = [Ctx() for _ in range(world)]
    layers = [DeviceLayer(c.ctx, cfg, owned=lambda e, r=r: bench.ep_owned(e, r, world)) for r, c in enumerate(ctxs)]
    try:
        x, _, _, resid = router_host_inputs(cfg)
        parts = torch.empty(world, 1, cfg.D, device="cuda")
        routes = None
        for r, (c, layer) in enumerate(zip(ctxs, layers)):
            xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
            ep = ExpertParallelLayer(c.ctx, r, world)
            idx = torch.empty(1, cfg.K, dtype=torch.int32, device="cuda")
            w = torch.empty(1, cfg.K, device="cuda")
            n = torch.empty(1, dtype=torch.int32, device="cuda")
            B.coli_router_select(c.ctx, xt, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale,
                                 idx, w, n)
            si, sw, sn = torch.empty_like(idx), torch.empty_like(w), torch.empty_like(n)
            B.coli_routes_shard(c.ctx, idx, w, n, r, world, si, sw, sn)
            B.coli_expert_group_issue(c.ctx, xt, si, sw, sn, cfg.K)
            B.coli_expert_group_take(c.ctx, None, parts[r])
            assert B.coli_check_error(c.ctx) == 0, B.coli_last_error(c.ctx)
            got = tuple(to_np(t) for t in (idx, w, n))
            if routes is None:
                routes = got
            else:  # every rank routes alike
                assert all(np.array_equal(a, b) for a, b in zip(got, routes))
            assert ep.world == world
        y = torch.empty(1, cfg.D, device="cuda")
        B.coli_partials_reduce(ctxs[0].ctx, parts, layers[0].act_tensor(resid), y)
        assert B.coli_check_error(ctxs[0].ctx) == 0
        idx, w, n = routes
        ref = O.ep_layer(x, oracle_experts(cfg, idx), idx, w, n, world, resid)
        assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), f"owned experts, world {world}")
    finally:
        for layer in layers:
            layer.free()
        for c in ctxs:
            c.close()
