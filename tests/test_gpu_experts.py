"""Grouped int4 expert FFN + weighted fixed-order reduce vs the oracle (small and ragged shapes)."""
import numpy as np
import pytest
import torch

import oracle.moe as O
from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from int4_grouped_expert_router_gb300.workload import CONFIGS, DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import (BF16_RTOL, F32_ATOL, F32_RTOL, Ctx, bf16_atol, f32_atol, assert_close, check_router, ffn_reference,
                      oracle_experts, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


def run_layer(ctx, cfg, token0=0, with_resid=True):
    layer = DeviceLayer(ctx, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg, token0)
        out = layer.outputs()
        layer.step(layer.act_tensor(x), layer.act_tensor(resid) if with_resid else None, out)
        assert B.coli_check_error(ctx) == 0
        idx, w, n, y = (to_np(out[k]) for k in ("idx", "w", "n_sel", "y"))
        near, _ = check_router(idx, w, n, x, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
        ref = ffn_reference(cfg, x, idx, w, n, resid if with_resid else None)
        return y, ref, near
    finally:
        layer.free()


def tol(cfg, ref):
    return (BF16_RTOL, bf16_atol(ref)) if cfg.x_dtype == "bf16" else (F32_RTOL, f32_atol(ref))


@pytest.mark.parametrize("cfg", [
    LayerConfig("tiny", D=256, I=128, E=16, K=4),
    LayerConfig("tiny-noresid", D=256, I=128, E=16, K=4),
    LayerConfig("g64", D=256, I=128, E=16, K=4, gs=64),
    LayerConfig("g32-mixed", D=256, I=128, E=16, K=4, gs="mixed:32"),
    LayerConfig("g64-tail", D=320, I=200, E=12, K=3, gs=64, topp=0.8),
    LayerConfig("ragged", D=200, I=136, E=20, K=5, gs=0),
    LayerConfig("generic-gs6", D=96, I=40, E=8, K=3, gs=6),
    LayerConfig("generic-gs2-mixed", D=64, I=34, E=8, K=2, gs="mixed:2"),
    LayerConfig("generic-gs48", D=256, I=100, E=8, K=4, gs=48),
    LayerConfig("topp", D=512, I=256, E=64, K=8, topp=0.7, norm_topk=True),
    LayerConfig("no-norm", D=256, I=128, E=32, K=6, norm_topk=False, routed_scale=1.0),
    LayerConfig("S3", D=256, I=128, E=16, K=4, S=3, topp=0.9),
    LayerConfig("S5-bf16", D=512, I=256, E=16, K=4, S=5, x_dtype="bf16", zipf=True),
    LayerConfig("S1-bf16", D=256, I=128, E=16, K=4, x_dtype="bf16"),
    LayerConfig("K16", D=128, I=64, E=64, K=16),
    # many kept routes: CTAs whose batch ranges span several routes
    LayerConfig("S9-36routes", D=256, I=136, E=24, K=4, S=9, topp=0.9, zipf=True),
    LayerConfig("S5K8-40routes-g64", D=320, I=200, E=32, K=8, S=5, gs="mixed:64"),
], ids=lambda c: c.name)
def test_layer_matches_oracle(ctx, cfg):
    y, ref, near = run_layer(ctx, cfg, with_resid=cfg.name != "tiny-noresid")
    assert near == 0
    rtol, atol = tol(cfg, ref)
    stats = assert_close(y, ref, rtol, atol, cfg.name)
    print(cfg.name, stats)


def test_given_routes_including_dropped_slots(ctx):
    cfg = LayerConfig("routes", D=256, I=128, E=10, K=4, S=2)
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        idx = np.array([[7, 2, -1, -1], [2, 9, 0, 3]], np.int32)
        w = np.array([[0.5, 1.25, 0, 0], [-0.75, 0.5, 2.0, 0.125]], np.float32)
        n = np.array([2, 4], np.int32)
        y = torch.empty(2, cfg.D, device="cuda")
        B.coli_expert_group(ctx, layer.act_tensor(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                            torch.from_numpy(n).cuda(), cfg.K, layer.act_tensor(resid), y)
        assert B.coli_check_error(ctx) == 0
        ref = ffn_reference(cfg, x, idx, w, n, resid)
        assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), "given routes")
        # n_sel NULL means every slot is kept
        idx2 = np.array([[1, 4, 5, 6], [0, 1, 2, 3]], np.int32)
        y2 = torch.empty(2, cfg.D, device="cuda")
        B.coli_expert_group(ctx, layer.act_tensor(x), torch.from_numpy(idx2).cuda(), torch.from_numpy(w).cuda(), None,
                            cfg.K, None, y2)
        assert B.coli_check_error(ctx) == 0
        ref2 = ffn_reference(cfg, x, idx2, w, np.array([4, 4]), None)
        assert_close(to_np(y2), ref2, F32_RTOL, f32_atol(ref2), "n_sel NULL")
    finally:
        layer.free()


def test_exact_integer_sums(ctx):
    """Integer activations and power-of-two scales make every gate/up dot product exact on both
    sides; the down projection is the identity, so y = SiLU(g) u row by row."""
    D, I = 64, 32
    q = lambda seed, r, c: ((synth.u64(seed, r * c) % np.uint64(16)).astype(np.int16) - 8).reshape(r, c)
    qg, qu = q(1, I, D), q(2, I, D)
    qd = np.zeros((D, I), np.int16)
    np.fill_diagonal(qd, 1)
    pg, pu, pd = O.pack_int4(qg), O.pack_int4(qu), O.pack_int4(qd)
    sg = np.full(I, 2.0 ** -4, np.float32)
    su = np.full(I, 2.0 ** -3, np.float32)
    sd = np.full(D, 1.0, np.float32)
    hs = [B.coli_expert_upload(ctx, torch.from_numpy(p), torch.from_numpy(s), r, c, 0)
          for p, s, r, c in ((pg, sg, I, D), (pu, su, I, D), (pd, sd, D, I))]
    B.coli_expert_table_set(ctx, 0, *hs)
    try:
        xi = ((synth.u64(3, D) % np.uint64(3)).astype(np.float32) - 1).reshape(1, D)
        y = torch.empty(1, D, device="cuda")
        B.coli_expert_group(ctx, torch.from_numpy(xi).cuda(), torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                            torch.ones(1, 1, device="cuda"), None, 1, None, y)
        assert B.coli_check_error(ctx) == 0
        yo = to_np(y)[0]
        ref = ffn_reference_single(pg, sg, pu, su, pd, sd, D, I, xi[0])
        assert_close(yo, ref, F32_RTOL, f32_atol(ref), "exact-integer")
        assert np.all(yo[I:] == 0.0)
    finally:
        B.coli_expert_table_set(ctx, 0, 0, 0, 0)
        for h in hs:
            B.coli_expert_free(ctx, h)


@pytest.mark.parametrize("D", [512, 1024], ids=["gemv-D512", "stream-D1024"])
def test_activation_outliers_dense_weights(ctx, D):
    """Massive-activation outliers (1e4 next to O(1) values in every 32-column chunk) with dense random
    weights: the case that stresses the block-fixed-point activations (each chunk is quantised relative to
    its outlier). y must meet the f32 tolerance, and its largest error may be at most four times that of a
    plain binary32 evaluation of the same sums (oracle.moe.expert_group_f32), which itself needs the
    rms-scaled absolute term here (output rms ~ 3e6)."""
    cfg = LayerConfig("outliers", D=D, I=256, E=8, K=4)
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        x[0, ::32] = 1.0e4 * np.sign(x[0, ::32] + 0.5)
        idx = np.array([[1, 5, 2, 7]], np.int32)
        w = np.array([[0.6, 0.25, 0.1, 0.05]], np.float32)
        y = torch.empty(1, cfg.D, device="cuda")
        B.coli_expert_group(ctx, layer.act_tensor(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), None,
                            cfg.K, layer.act_tensor(resid), y)
        assert B.coli_check_error(ctx) == 0
        experts = oracle_experts(cfg, idx)
        ref = O.expert_group(x, experts, idx, w, np.array([4]), resid)
        f32err = float(np.abs(O.expert_group_f32(x, experts, idx, w, np.array([4]), resid) - ref).max())
        stats = assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), "outliers")
        print("outliers", D, stats, "plain-f32 max err", f32err)
        assert stats["max_abs"] <= 4 * f32err, (stats["max_abs"], f32err)
    finally:
        layer.free()


def ffn_reference_single(pg, sg, pu, su, pd, sd, D, I, x):
    return O.expert_ffn(x, O.Tensor(pg, sg, I, D, 0), O.Tensor(pu, su, I, D, 0), O.Tensor(pd, sd, D, I, 0))


def test_deterministic_bits(ctx):
    cfg = LayerConfig("det", D=512, I=256, E=32, K=8, gs="mixed:64", topp=0.9)
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        ys = []
        for _ in range(4):
            out = layer.outputs()
            layer.step(layer.act_tensor(x), layer.act_tensor(resid), out)
            ys.append(out["y"].cpu().numpy().tobytes() + out["w"].cpu().numpy().tobytes() + out["idx"].cpu().numpy().tobytes())
        assert all(v == ys[0] for v in ys)
    finally:
        layer.free()


def test_bad_route_sets_error_word(ctx):
    cfg = LayerConfig("bad", D=128, I=64, E=4, K=2)
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, _ = router_host_inputs(cfg)
        y = torch.empty(1, cfg.D, device="cuda")
        for bad in (5, 4095, 100000, -3):
            idx = torch.tensor([[1, bad]], dtype=torch.int32, device="cuda")
            B.coli_expert_group(ctx, layer.act_tensor(x), idx, torch.ones(1, 2, device="cuda"), None, 2, None, y)
            assert B.coli_check_error(ctx) == B.COLI_E_ROUTE, bad
        # the context stays healthy
        idx = torch.tensor([[1, 2]], dtype=torch.int32, device="cuda")
        B.coli_expert_group(ctx, layer.act_tensor(x), idx, torch.ones(1, 2, device="cuda"), None, 2, None, y)
        assert B.coli_check_error(ctx) == 0
    finally:
        layer.free()
