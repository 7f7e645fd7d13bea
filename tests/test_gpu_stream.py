"""S = 1 decode through the streaming FFN (the down projection split by 16-row units, a fixed-order
reduce of per-CTA partial rows) against the oracle, against the two-kernel form, and its bounded waits.

The streaming kernel runs when D is a multiple of 1024 (up to 6144), I a multiple of 16 and every
table entry has per-row or 32-multiple group scales; the profile then records one gate/up-kind
launch (the streaming kernel), one combine-kind launch (its reduce) and no down launch per call.
"""
import os

import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import BF16_RTOL, F32_RTOL, Ctx, assert_close, bf16_atol, check_router, f32_atol, ffn_reference, to_np

pytestmark = pytest.mark.gpu


def make_ctx(**env) -> Ctx:
    old = {k: os.environ.get(k) for k in env}
    os.environ.update({k: str(v) for k, v in env.items()})
    try:
        return Ctx()
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


@pytest.fixture(scope="module")
def ctxs():
    cs, c2 = make_ctx(COLI_DECODE_STREAM=1), make_ctx(COLI_DECODE_STREAM=0)
    yield cs.ctx, c2.ctx
    cs.close()
    c2.close()


def launches(ctx):
    return tuple(B.coli_profile_read(ctx, k)[1] for k in (B.COLI_KERNEL_GATEUP, B.COLI_KERNEL_DOWN))


CASES = [
    LayerConfig("D1024-row", D=1024, I=128, E=16, K=4),
    LayerConfig("D1024-g64", D=1024, I=128, E=16, K=4, gs=64),
    LayerConfig("D2048-g32-mixed", D=2048, I=256, E=16, K=4, gs="mixed:32"),
    # I a multiple of 16 but not of 32; a g64 tail group of 16 columns in the down rows
    LayerConfig("D1024-I208-g64-tail-topp", D=1024, I=208, E=12, K=3, gs=64, topp=0.8),
    LayerConfig("D3072-topp-K8", D=3072, I=512, E=64, K=8, topp=0.7),
    LayerConfig("D1024-K16", D=1024, I=64, E=64, K=16),
    LayerConfig("D2048-bf16", D=2048, I=256, E=16, K=4, x_dtype="bf16"),
    LayerConfig("D1024-no-norm", D=1024, I=96, E=32, K=6, norm_topk=False, routed_scale=1.0),
    # fewer units than CTAs; D = 7168 (two stages of each ring no longer fit) takes the two-kernel form
    LayerConfig("D5120-I64", D=5120, I=64, E=8, K=2),
    # more units than CTAs on one slot, CTAs spanning slots, g96 groups (D % gs != 0 for the gate rows)
    LayerConfig("D6144-I1024-g96", D=6144, I=1024, E=8, K=3, gs=96),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_stream_matches_oracle_and_two_kernel_form(ctxs, cfg):
    cs, c2 = ctxs
    ls, l2 = DeviceLayer(cs, cfg), DeviceLayer(c2, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg)
        B.coli_profile_enable(cs, 1)
        launches(cs)
        os_, o2 = ls.outputs(), l2.outputs()
        xt, rt = ls.act_tensor(x), ls.act_tensor(resid)
        ls.step(xt, rt, os_)
        l2.step(l2.act_tensor(x), l2.act_tensor(resid), o2)
        assert B.coli_check_error(cs) == 0, B.coli_last_error(cs)
        assert B.coli_check_error(c2) == 0, B.coli_last_error(c2)
        assert launches(cs) == (1, 0)  # the whole FFN in one streaming launch (plus its reduce)
        B.coli_profile_enable(cs, 0)
        for k in ("idx", "w", "n_sel"):
            assert torch.equal(os_[k], o2[k]), k
        idx, w, n, y = (to_np(os_[k]) for k in ("idx", "w", "n_sel", "y"))
        near, _ = check_router(idx, w, n, x, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
        assert near == 0
        ref = ffn_reference(cfg, to_np(xt), idx, w, n, to_np(rt))
        if cfg.x_dtype == "bf16":
            assert_close(y, ref, BF16_RTOL, bf16_atol(ref), cfg.name)
            assert_close(to_np(o2["y"]), y, BF16_RTOL, bf16_atol(ref), cfg.name + " vs two-kernel")
        else:
            stats = assert_close(y, ref, F32_RTOL, f32_atol(ref), cfg.name)
            assert_close(to_np(o2["y"]), y, 2 * F32_RTOL, 2 * f32_atol(ref), cfg.name + " vs two-kernel")
            print(cfg.name, stats)
        # bit-identical from run to run
        y0 = os_["y"].clone()
        for _ in range(3):
            ls.step(xt, rt, os_)
            assert torch.equal(os_["y"], y0)
        assert B.coli_check_error(cs) == 0
    finally:
        ls.free()
        l2.free()


def test_stream_given_routes_dropped_and_repeated_slots(ctxs):
    """Routes given by hand: dropped slots (n_sel < K), the same expert in two slots, no residual."""
    cs, _ = ctxs
    cfg = LayerConfig("given", D=2048, I=128, E=8, K=5, gs="mixed:64")
    layer = DeviceLayer(cs, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        idx = np.array([[3, 3, 6, -1, -1]], np.int32)
        w = np.array([[0.7, -0.25, 1.5, 0.0, 0.0]], np.float32)
        n = np.array([3], np.int32)
        xt = layer.act_tensor(x)
        y = torch.empty(1, cfg.D, device="cuda")
        for r in (resid, None):
            rt = layer.act_tensor(r) if r is not None else None
            B.coli_expert_group(cs, xt, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                                torch.from_numpy(n).cuda(), cfg.K, rt, y)
            assert B.coli_check_error(cs) == 0, B.coli_last_error(cs)
            ref = ffn_reference(cfg, x, idx, w, n, r)
            assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), "given routes")
        # every slot dropped: y = residual exactly
        n0 = torch.zeros(1, dtype=torch.int32, device="cuda")
        rt = layer.act_tensor(resid)
        B.coli_expert_group(cs, xt, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), n0, cfg.K, rt, y)
        assert B.coli_check_error(cs) == 0
        assert torch.equal(y, rt)
    finally:
        layer.free()


def test_stream_bad_route_then_healthy(ctxs):
    cs, _ = ctxs
    cfg = LayerConfig("bad", D=1024, I=64, E=8, K=2)
    layer = DeviceLayer(cs, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        y = torch.empty(1, cfg.D, device="cuda")
        bad = torch.tensor([[2, 4000]], dtype=torch.int32, device="cuda")  # 4000: an unset table entry
        w = torch.tensor([[0.5, 0.5]], device="cuda")
        B.coli_expert_group(cs, xt, bad, w, None, cfg.K, rt, y)
        assert B.coli_check_error(cs) == B.COLI_E_ROUTE
        good = torch.tensor([[2, 5]], dtype=torch.int32, device="cuda")
        B.coli_expert_group(cs, xt, good, w, None, cfg.K, rt, y)
        assert B.coli_check_error(cs) == 0
        ref = ffn_reference(cfg, x, good.cpu().numpy(), w.cpu().numpy(), None, resid)
        assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), "after a bad route")
    finally:
        layer.free()


def test_stream_bounded_wait_gives_up_then_healthy():
    """One CTA's producer withholds the copy of its first stage (test hook, one launch): the waits on that
    stage give up after the shortened limit, the waits behind them too, and the call reports
    COLI_E_TIMEOUT; the next call is healthy and matches the oracle. No wait is unbounded and nothing
    traps."""
    c = make_ctx(COLI_DECODE_STREAM=1, COLI_TEST_WAIT_NS=20_000_000, COLI_TEST_WITHHOLD=1)
    cfg = LayerConfig("timeout", D=1024, I=64, E=8, K=2)
    layer = DeviceLayer(c.ctx, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        out = layer.outputs()
        layer.step(xt, rt, out)
        assert B.coli_check_error(c.ctx) == B.COLI_E_TIMEOUT
        layer.step(xt, rt, out)
        assert B.coli_check_error(c.ctx) == 0, B.coli_last_error(c.ctx)
        idx, w, n, y = (to_np(out[k]) for k in ("idx", "w", "n_sel", "y"))
        ref = ffn_reference(cfg, x, idx, w, n, resid)
        assert_close(y, ref, F32_RTOL, f32_atol(ref), "after a timeout")
    finally:
        layer.free()
        c.close()
