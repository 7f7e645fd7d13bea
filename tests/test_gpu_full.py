"""Full-shape decode layers (D=6144, I=2048 or 2000, E=256, K=8) against the oracle on sampled tokens,
in the launch configuration the benchmark times."""
import numpy as np
import torch
import pytest

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.workload import CONFIGS, DeviceLayer, router_host_inputs
from gpu_util import BF16_RTOL, F32_ATOL, F32_RTOL, Ctx, bf16_atol, f32_atol, assert_close, check_router, ffn_reference, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


@pytest.mark.parametrize("name,tokens", [("decode", (0, 1, 2)), ("decode_g64", (0, 1)), ("decode_g64_tail", (0,)),
                                         ("decode_s4_bf16", (0,))])
def test_full_shape_layer(ctx, name, tokens):
    cfg = CONFIGS[name]
    layer = DeviceLayer(ctx, cfg)
    try:
        for tok in tokens:
            x, Wr, bias, resid = router_host_inputs(cfg, tok)
            out = layer.outputs()
            layer.step(layer.act_tensor(x), layer.act_tensor(resid), out)
            assert B.coli_check_error(ctx) == 0
            idx, w, n, y = (to_np(out[k]) for k in ("idx", "w", "n_sel", "y"))
            near, werr = check_router(idx, w, n, x, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
            ref = ffn_reference(cfg, x, idx, w, n, resid)
            if cfg.x_dtype == "bf16":
                stats = assert_close(y, ref, BF16_RTOL, bf16_atol(ref), name)
            else:
                stats = assert_close(y, ref, F32_RTOL, f32_atol(ref), name)
            print(name, tok, "near-ties", near, "distinct", len(set(idx[idx >= 0].tolist())), stats)
            assert near <= 1
    finally:
        layer.free()


def test_full_shape_prefill_tensor_core_path(ctx):
    """S=512 tokens, g64 int4, bf16, Zipf routing: the tensor-core path. Router checked on every
    token; the FFN on sampled tokens (bf16 tensor-core tolerance: see test_gpu_prefill)."""
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
        sel = [0, 137, 511]
        ref = ffn_reference(cfg, xb[sel], idx[sel], w[sel], n[sel], rb[sel])
        stats = assert_close(y[sel], ref, TC_RTOL, tc_atol(ref), "prefill")
        assert stats["norm_rel"] < TC_NORM, stats
        print("prefill near-ties", near, "experts touched", int((rows > 0).sum()), "max rows", int(rows.max()), stats)
    finally:
        layer.free()
