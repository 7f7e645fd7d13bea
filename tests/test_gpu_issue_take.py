"""Resident issue/take (PR #434 "COLI_CUDA_RESID=1", section "What"): issued groups' partial sums stay on
the device and one take joins them, in issue order, to the residual.

- One issue holding all of a token's routes gives y bit-identical to coli_expert_group, on the GEMV paths (S = 1,
  S > 1) and on the tensor-core path.
- Routes split into several issues give resid + (p_0 + p_1 + ...) exactly, each p_j taken from its own round, and
  stay within the oracle's tolerance.
- Router, issue and take captured in one CUDA graph replay to the same bits as the eager calls.
- A take with nothing issued, more than COLI_MAX_ISSUES issues, or a round whose issues disagree on S is rejected,
  and the context stays usable.
"""
import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import F32_RTOL, Ctx, assert_close, f32_atol, ffn_reference, to_np

pytestmark = pytest.mark.gpu

COLI_MAX_ISSUES = B.COLI_MAX_ISSUES


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


def route(layer, x):
    out = layer.outputs(x.shape[0])
    c = layer.cfg
    B.coli_router_select(layer.ctx, x, layer.Wr, layer.bias, c.K, c.topp, c.norm_topk, c.routed_scale,
                         out["idx"], out["w"], out["n_sel"])
    return out


@pytest.mark.parametrize("cfg", [
    LayerConfig("S1-f32", D=256, I=128, E=16, K=4),
    LayerConfig("S1-topp-g64", D=320, I=200, E=12, K=3, gs=64, topp=0.8),
    LayerConfig("S1-bf16", D=256, I=128, E=16, K=4, x_dtype="bf16"),
    LayerConfig("S5-bf16", D=512, I=256, E=16, K=4, S=5, x_dtype="bf16", zipf=True),
    LayerConfig("S3-f32", D=256, I=128, E=16, K=4, S=3, topp=0.9),
    # S K = 256 routed rows over 16 experts: the tensor-core path
    LayerConfig("tc-S64", D=256, I=128, E=16, K=4, S=64, gs=64, x_dtype="bf16", zipf=True),
], ids=lambda c: c.name)
def test_single_issue_equals_expert_group(ctx, cfg):
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        r = route(layer, xt)
        y_sync = torch.empty_like(xt)
        B.coli_expert_group(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K, rt, y_sync)
        assert B.coli_expert_group_issue(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K) == 0
        y = torch.empty_like(xt)
        B.coli_expert_group_take(ctx, rt, y)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        assert torch.equal(y, y_sync), (y.float() - y_sync.float()).abs().max()
    finally:
        layer.free()


def split_routes(idx, w, n, k0):
    """Slots [0, k0) and [k0, K) of every token as two groups, each with its own kept count."""
    K = idx.shape[1]
    ga = (idx[:, :k0].contiguous(), w[:, :k0].contiguous(), torch.clamp(n, max=k0).to(torch.int32).contiguous())
    gb = (idx[:, k0:].contiguous(), w[:, k0:].contiguous(), torch.clamp(n - k0, min=0).to(torch.int32).contiguous())
    return (ga, k0), (gb, K - k0)


@pytest.mark.parametrize("cfg", [
    LayerConfig("split-S1", D=256, I=128, E=16, K=6),
    LayerConfig("split-S4-topp", D=320, I=200, E=20, K=5, S=4, gs="mixed:64", topp=0.85),
], ids=lambda c: c.name)
def test_split_issues_sum_in_issue_order(ctx, cfg):
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        r = route(layer, xt)
        groups = split_routes(r["idx"], r["w"], r["n_sel"], 2)
        # each group's partial sum on its own (one issue, no residual)
        parts = []
        for (gi, gw, gn), k in groups:
            assert B.coli_expert_group_issue(ctx, xt, gi, gw, gn, k) == 0
            p = torch.empty_like(xt)
            B.coli_expert_group_take(ctx, None, p)
            parts.append(to_np(p))
        # both groups in one round
        for j, ((gi, gw, gn), k) in enumerate(groups):
            assert B.coli_expert_group_issue(ctx, xt, gi, gw, gn, k) == j
        y = torch.empty_like(xt)
        B.coli_expert_group_take(ctx, rt, y)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        expect = to_np(rt).astype(np.float32) + (parts[0].astype(np.float32) + parts[1].astype(np.float32))
        assert np.array_equal(to_np(y), expect)
        ref = ffn_reference(cfg, x, to_np(r["idx"]), to_np(r["w"]), to_np(r["n_sel"]), resid)
        print(cfg.name, assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), cfg.name))
    finally:
        layer.free()


def test_graph_captured_layer(ctx):
    """Router + issue + take as one CUDA graph: replays match the eager calls bit for bit."""
    cfg = LayerConfig("graph", D=512, I=256, E=32, K=8, topp=0.9)
    layer = DeviceLayer(ctx, cfg)
    stream = torch.cuda.Stream()
    B.coli_set_stream(ctx, stream)
    try:
        B.coli_reserve(ctx, cfg.S, cfg.E, cfg.K, cfg.D, cfg.I)
        xin = torch.empty(cfg.S, cfg.D, device="cuda")
        rin = torch.empty_like(xin)
        yout = torch.empty_like(xin)
        r = layer.outputs()

        def body():
            B.coli_router_select(ctx, xin, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale,
                                 r["idx"], r["w"], r["n_sel"])
            B.coli_expert_group_issue(ctx, xin, r["idx"], r["w"], r["n_sel"], cfg.K)
            B.coli_expert_group_take(ctx, rin, yout)

        with torch.cuda.stream(stream):
            xin.copy_(layer.act_tensor(router_host_inputs(cfg, 0)[0]))
            rin.copy_(layer.act_tensor(router_host_inputs(cfg, 0)[3]))
            body()  # eager once: the workspace and the slot pool exist before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        for tok in range(1, 4):
            x, _, _, resid = router_host_inputs(cfg, tok)
            with torch.cuda.stream(stream):
                xin.copy_(layer.act_tensor(x))
                rin.copy_(layer.act_tensor(resid))
                g.replay()
            torch.cuda.synchronize()
            y_graph = yout.clone()
            with torch.cuda.stream(stream):
                ref = layer.outputs()
                layer.step(xin, rin, ref)  # the two synchronous calls, eager
            assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
            assert torch.equal(r["idx"], ref["idx"])
            assert torch.equal(y_graph, ref["y"]), tok
    finally:
        B.coli_set_stream(ctx, torch.cuda.current_stream())
        layer.free()


def test_rejected_rounds_leave_context_usable(ctx):
    cfg = LayerConfig("limits", D=128, I=64, E=8, K=2)
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        r = route(layer, xt)
        y = torch.empty_like(xt)
        with pytest.raises(B.ColiError) as e:
            B.coli_expert_group_take(ctx, rt, y)
        assert e.value.code == B.COLI_E_INVAL
        # COLI_MAX_ISSUES pending, the next one refused, the take sums all of them
        for j in range(COLI_MAX_ISSUES):
            assert B.coli_expert_group_issue(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K) == j
        with pytest.raises(B.ColiError) as e:
            B.coli_expert_group_issue(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K)
        assert e.value.code == B.COLI_E_INVAL
        B.coli_expert_group_take(ctx, None, y)
        one = torch.empty_like(xt)
        B.coli_expert_group_issue(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K)
        B.coli_expert_group_take(ctx, None, one)
        acc = to_np(one).astype(np.float32)
        p = acc.copy()
        for _ in range(COLI_MAX_ISSUES - 1):
            acc = (acc + p).astype(np.float32)
        assert np.array_equal(to_np(y), acc)
        # a round's issues must agree on S
        x2 = torch.cat([xt, xt])
        B.coli_expert_group_issue(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K)
        with pytest.raises(B.ColiError) as e:
            B.coli_expert_group_issue(ctx, x2, r["idx"].repeat(2, 1), r["w"].repeat(2, 1), r["n_sel"].repeat(2), cfg.K)
        assert e.value.code == B.COLI_E_INVAL
        B.coli_expert_group_take(ctx, rt, y)
        y_sync = torch.empty_like(xt)
        B.coli_expert_group(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K, rt, y_sync)
        assert B.coli_check_error(ctx) == 0
        assert torch.equal(y, y_sync)
    finally:
        layer.free()
