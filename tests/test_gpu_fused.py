"""S = 1 decode: the one-kernel (cooperative, opt-in) expert FFN against the two-kernel form and the oracle.

Both forms share the dot-product, slice-sum and slot-order reduce arithmetic, so y must agree bit
for bit; the fused form is checked to be the one that ran (one kernel per call, none recorded as
down). Repeated calls check that the kernel's cross-CTA counters are left ready for the next call.
"""
import os

import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import BF16_RTOL, F32_RTOL, Ctx, assert_close, bf16_atol, check_router, f32_atol, ffn_reference, to_np

pytestmark = pytest.mark.gpu


def make_ctx(fused: bool) -> Ctx:
    old = os.environ.get("COLI_DECODE_FUSED")
    os.environ["COLI_DECODE_FUSED"] = "1" if fused else "0"
    try:
        return Ctx()
    finally:
        if old is None:
            del os.environ["COLI_DECODE_FUSED"]
        else:
            os.environ["COLI_DECODE_FUSED"] = old


@pytest.fixture(scope="module")
def ctxs():
    cf, c2 = make_ctx(True), make_ctx(False)
    yield cf.ctx, c2.ctx
    cf.close()
    c2.close()


def launches(ctx):
    return tuple(B.coli_profile_read(ctx, k)[1] for k in (B.COLI_KERNEL_GATEUP, B.COLI_KERNEL_DOWN))


CASES = [
    LayerConfig("tiny", D=256, I=128, E=16, K=4),
    LayerConfig("g64", D=256, I=128, E=16, K=4, gs=64),
    LayerConfig("g32-mixed", D=256, I=128, E=16, K=4, gs="mixed:32"),
    LayerConfig("g64-tail-topp", D=320, I=200, E=12, K=3, gs=64, topp=0.8),
    LayerConfig("ragged", D=200, I=136, E=20, K=5),
    LayerConfig("generic-gs6", D=96, I=40, E=8, K=3, gs=6),
    LayerConfig("topp", D=512, I=256, E=64, K=8, topp=0.7),
    LayerConfig("K16", D=128, I=64, E=64, K=16),
    LayerConfig("bf16", D=256, I=128, E=16, K=4, x_dtype="bf16"),
    # four column slices per down row (the widest fused form), D not a multiple of the row batch
    LayerConfig("I4096", D=198, I=4096, E=8, K=4, gs="mixed:64"),
    # K * slices streams above the row ranges of a small D
    LayerConfig("K32-I2048", D=64, I=2048, E=40, K=32),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_fused_matches_two_kernel_form_and_oracle(ctxs, cfg):
    cf, c2 = ctxs
    lf, l2 = DeviceLayer(cf, cfg), DeviceLayer(c2, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg)
        B.coli_profile_enable(cf, 1)
        launches(cf)
        of, o2 = lf.outputs(), l2.outputs()
        lf.step(lf.act_tensor(x), lf.act_tensor(resid), of)
        l2.step(l2.act_tensor(x), l2.act_tensor(resid), o2)
        assert B.coli_check_error(cf) == 0, B.coli_last_error(cf)
        assert B.coli_check_error(c2) == 0, B.coli_last_error(c2)
        assert launches(cf) == (1, 0)  # one kernel for the whole FFN
        B.coli_profile_enable(cf, 0)
        for k in ("idx", "w", "n_sel"):
            assert torch.equal(of[k], o2[k]), k
        assert torch.equal(of["y"], o2["y"]), (of["y"] - o2["y"]).abs().max()
        idx, w, n, y = (to_np(of[k]) for k in ("idx", "w", "n_sel", "y"))
        xw, rw = to_np(lf.act_tensor(x)), to_np(lf.act_tensor(resid))
        near, _ = check_router(idx, w, n, xw, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
        assert near == 0
        ref = ffn_reference(cfg, xw, idx, w, n, rw)
        rtol, atol = (BF16_RTOL, bf16_atol(ref)) if cfg.x_dtype == "bf16" else (F32_RTOL, f32_atol(ref))
        print(cfg.name, assert_close(y, ref, rtol, atol, cfg.name))
        for _ in range(3):  # counters and barrier left ready: same bits every call
            lf.step(lf.act_tensor(x), lf.act_tensor(resid), of)
            assert B.coli_check_error(cf) == 0
            assert torch.equal(of["y"], o2["y"])
    finally:
        lf.free()
        l2.free()


def test_fused_wide_rows_fall_back(ctxs):
    """I above the fused form's four column slices: separate gate/up and down kernels."""
    cf, _ = ctxs
    cfg = LayerConfig("I4160", D=64, I=4160, E=4, K=2)
    layer = DeviceLayer(cf, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        B.coli_profile_enable(cf, 1)
        launches(cf)
        out = layer.outputs()
        layer.step(layer.act_tensor(x), layer.act_tensor(resid), out)
        assert B.coli_check_error(cf) == 0
        assert launches(cf) == (1, 1)
        B.coli_profile_enable(cf, 0)
        idx, w, n, y = (to_np(out[k]) for k in ("idx", "w", "n_sel", "y"))
        ref = ffn_reference(cfg, x, idx, w, n, resid)
        assert_close(y, ref, F32_RTOL, f32_atol(ref), cfg.name)
    finally:
        layer.free()


def test_fused_given_routes(ctxs):
    """Dropped slots, invalid slots beyond n_sel, no kept slot at all (y = residual), NULL n_sel."""
    cf, c2 = ctxs
    cfg = LayerConfig("routes", D=256, I=128, E=10, K=4)
    lf, l2 = DeviceLayer(cf, cfg), DeviceLayer(c2, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        cases = [
            (np.array([[7, 2, -1, -1]], np.int32), np.array([2], np.int32)),
            (np.array([[3, -5, 4095, 9]], np.int32), np.array([1], np.int32)),
            (np.array([[-1, -1, -1, -1]], np.int32), np.array([0], np.int32)),
            (np.array([[1, 4, 5, 6]], np.int32), None),
        ]
        w = torch.tensor([[0.5, 1.25, -0.75, 2.0]], device="cuda")
        for idx, n in cases:
            ys = []
            for ctx, layer in ((cf, lf), (c2, l2)):
                y = torch.empty(1, cfg.D, device="cuda")
                B.coli_expert_group(ctx, layer.act_tensor(x), torch.from_numpy(idx).cuda(), w,
                                    None if n is None else torch.from_numpy(n).cuda(), cfg.K, layer.act_tensor(resid), y)
                assert B.coli_check_error(ctx) == 0, (idx, B.coli_last_error(ctx))
                ys.append(y)
            assert torch.equal(ys[0], ys[1]), idx
            nn = np.array([4], np.int32) if n is None else n
            ref = ffn_reference(cfg, x, idx, w.cpu().numpy(), nn, resid)
            assert_close(to_np(ys[0]), ref, F32_RTOL, f32_atol(ref), str(idx))
            if n is not None and n[0] == 0:
                assert torch.equal(ys[0], lf.act_tensor(resid))
    finally:
        lf.free()
        l2.free()


def test_fused_bad_route_then_healthy(ctxs):
    """An unset table entry among the kept slots sets COLI_E_ROUTE; the next call is clean and exact."""
    cf, c2 = ctxs
    cfg = LayerConfig("bad", D=128, I=64, E=4, K=2)
    lf, l2 = DeviceLayer(cf, cfg), DeviceLayer(c2, cfg)
    try:
        x, _, _, _ = router_host_inputs(cfg)
        y = torch.empty(1, cfg.D, device="cuda")
        for bad in (5, 4095, -3):
            idx = torch.tensor([[1, bad]], dtype=torch.int32, device="cuda")
            B.coli_expert_group(cf, lf.act_tensor(x), idx, torch.ones(1, 2, device="cuda"), None, 2, None, y)
            assert B.coli_check_error(cf) == B.COLI_E_ROUTE, bad
        idx = torch.tensor([[1, 2]], dtype=torch.int32, device="cuda")
        y2 = torch.empty_like(y)
        B.coli_expert_group(cf, lf.act_tensor(x), idx, torch.ones(1, 2, device="cuda"), None, 2, None, y)
        B.coli_expert_group(c2, l2.act_tensor(x), idx, torch.ones(1, 2, device="cuda"), None, 2, None, y2)
        assert B.coli_check_error(cf) == 0 and B.coli_check_error(c2) == 0
        assert torch.equal(y, y2)
    finally:
        lf.free()
        l2.free()
