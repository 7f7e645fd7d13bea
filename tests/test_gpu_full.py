"""Full-shape decode layers (D=6144, I=2048 or 2000, E=256, K=8) against the oracle on sampled tokens,
in the launch configuration the benchmark times."""
import numpy as np
import torch
import pytest

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.workload import CONFIGS, DeviceLayer, router_host_inputs
from gpu_util import (BF16_RTOL, F32_ATOL, F32_RTOL, Ctx, bf16_atol, f32_atol, assert_close, check_router, ffn_reference,
                      oracle_experts, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


@pytest.mark.parametrize("name,tokens", [("decode", range(16)), ("decode_g64", range(8)), ("decode_g64_tail", range(8)),
                                         ("decode_s4_bf16", range(4))])
def test_full_shape_layer(ctx, name, tokens):
    """Every sampled token is checked element by element. f32 tokens are also held to the accuracy of a plain
    binary32 evaluation of the oracle's sums (oracle.moe.expert_group_f32): the GPU's largest error may be at
    most twice that evaluation's."""
    import oracle.moe as O
    cfg = CONFIGS[name]
    layer = DeviceLayer(ctx, cfg)
    try:
        worst = 0.0
        for tok in tokens:
            x, Wr, bias, resid = router_host_inputs(cfg, tok)
            out = layer.outputs()
            layer.step(layer.act_tensor(x), layer.act_tensor(resid), out)
            assert B.coli_check_error(ctx) == 0
            idx, w, n, y = (to_np(out[k]) for k in ("idx", "w", "n_sel", "y"))
            near, werr = check_router(idx, w, n, x, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
            experts = oracle_experts(cfg, idx)
            ref = O.expert_group(x, experts, idx, w, n, resid)
            if cfg.x_dtype == "bf16":
                stats = assert_close(y, ref, BF16_RTOL, bf16_atol(ref), name)
                f32err = None
            else:
                stats = assert_close(y, ref, F32_RTOL, f32_atol(ref), name)
                f32err = float(np.abs(O.expert_group_f32(x, experts, idx, w, n, resid) - ref).max())
                assert stats["max_abs"] <= 2 * f32err, (stats["max_abs"], f32err)
            worst = max(worst, stats["max_abs"] / (f32_atol(ref) if cfg.x_dtype != "bf16" else bf16_atol(ref)))
            print(name, tok, "near-ties", near, "distinct", len(set(idx[idx >= 0].tolist())), stats,
                  "plain-f32 max err", f32err)
            assert near <= 1
        print(name, "worst |err| / abs term", round(worst, 3))
    finally:
        layer.free()


def test_full_shape_prefill_tensor_core_path(ctx):
    """S=512 tokens, g64 int4, bf16, Zipf routing: the tensor-core path. Router checked on every
    token; the FFN on 32 tokens spread over the entry sizes (bf16 tensor-core tolerance: see
    test_gpu_prefill); every token's output is checked for run-to-run bit identity."""
    from test_gpu_prefill import TC_NORM, TC_RTOL, tc_atol

    cfg = CONFIGS["prefill"]
    layer = DeviceLayer(ctx, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg, 7)
        out = layer.outputs()
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        layer.step(xt, rt, out)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        y0 = out["y"].clone()
        for _ in range(4):  # bit-identical from run to run at full size (every token, every column)
            layer.step(xt, rt, out)
            assert B.coli_check_error(ctx) == 0
            assert torch.equal(out["y"], y0), int((out["y"] != y0).sum())
        idx, w, n, y = (to_np(out[k]) for k in ("idx", "w", "n_sel", "y"))
        xb, rb = to_np(xt), to_np(rt)
        near, _ = check_router(idx, w, n, xb, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
        assert near <= 3
        rows = np.bincount(idx[idx >= 0].reshape(-1), minlength=cfg.E)
        # 32 tokens spread over the entry-size classes: ranked by the smallest routed row count among their
        # kept experts (experts of one entry, of several entries of 128 rows, and between), evenly sampled
        small = np.array([rows[idx[t][idx[t] >= 0]].min() for t in range(cfg.S)])
        order = np.argsort(small, kind="stable")
        sel = sorted(set(order[np.linspace(0, cfg.S - 1, 32).astype(int)].tolist()))
        ref = ffn_reference(cfg, xb[sel], idx[sel], w[sel], n[sel], rb[sel])
        stats = assert_close(y[sel], ref, TC_RTOL, tc_atol(ref), "prefill")
        assert stats["norm_rel"] < TC_NORM, stats
        print("prefill near-ties", near, "experts touched", int((rows > 0).sum()), "max rows", int(rows.max()),
              "checked tokens", len(sel), "smallest-row classes", sorted(set(small[sel].tolist())), stats)
    finally:
        layer.free()
