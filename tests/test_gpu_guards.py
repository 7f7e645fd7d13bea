"""Guard words around every output buffer: each output is a view into a larger buffer whose elements
before and after it hold a sentinel bit pattern; after each call the sentinels must be unchanged (no
write lands outside the output), and the outputs must still match the oracle.

The shapes are the ragged ones: D = 7000 (rows of 3500 bytes, no whole number of 16-byte chunks),
I = 200, the 16-column tail group of I = 2000 on the streaming path, and bf16 rows of D = 200 that are
not 16-byte aligned (S = 3).
"""
import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import BF16_RTOL, F32_RTOL, Ctx, assert_close, bf16_atol, check_router, f32_atol, ffn_reference, to_np

pytestmark = pytest.mark.gpu

GUARD = 257  # elements of sentinel on each side (an odd count: the views start off any 16-byte boundary)


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


def guarded(shape, dtype):
    """(buffer, view): the view has `shape` and sits between GUARD sentinel elements on each side."""
    n = int(np.prod(shape))
    if dtype == torch.int32:
        buf = torch.full((n + 2 * GUARD,), -0x21524111, dtype=torch.int32, device="cuda")  # 0xDEADBEEF
    elif dtype == torch.float32:
        buf = torch.full((n + 2 * GUARD,), 0, dtype=torch.int32, device="cuda").fill_(0x7FBADBAD).view(torch.float32)
    else:
        buf = torch.full((n + 2 * GUARD,), 0, dtype=torch.int16, device="cuda").fill_(0x7FBD).view(torch.bfloat16)
    return buf, buf[GUARD:GUARD + n].view(shape)


def intact(buf, n):
    b = buf.view(torch.int16 if buf.dtype == torch.bfloat16 else torch.int32)
    ref = {torch.bfloat16: 0x7FBD, torch.float32: 0x7FBADBAD, torch.int32: -0x21524111}[buf.dtype]
    head, tail = b[:GUARD], b[GUARD + n:]
    return bool((head == ref).all()) and bool((tail == ref).all())


CASES = [
    LayerConfig("D7000-I200", D=7000, I=200, E=12, K=4),
    LayerConfig("D7000-I200-g64", D=7000, I=200, E=12, K=4, gs="mixed:64", topp=0.8),
    LayerConfig("D6144-I2000-g64-tail-stream", D=6144, I=2000, E=8, K=4, gs=64),
    LayerConfig("S3-D200-bf16", D=200, I=136, E=12, K=3, S=3, x_dtype="bf16"),
    LayerConfig("S3-D7000-I200", D=7000, I=200, E=12, K=4, S=3, topp=0.9),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_outputs_are_written_only_inside_their_buffers(ctx, cfg):
    layer = DeviceLayer(ctx, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        dt = torch.bfloat16 if cfg.x_dtype == "bf16" else torch.float32
        bi, idx = guarded((cfg.S, cfg.K), torch.int32)
        bw, w = guarded((cfg.S, cfg.K), torch.float32)
        bn, n = guarded((cfg.S,), torch.int32)
        by, y = guarded((cfg.S, cfg.D), dt)
        for call in range(2):
            B.coli_router_select(ctx, xt, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale,
                                 idx, w, n)
            B.coli_expert_group(ctx, xt, idx, w, n, cfg.K, rt, y)
            assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
            for buf, view in ((bi, idx), (bw, w), (bn, n), (by, y)):
                assert intact(buf, view.numel()), (call, buf.dtype)
        xh, rh = to_np(xt), to_np(rt)
        ih, wh, nh, yh = to_np(idx), to_np(w), to_np(n), to_np(y)
        near, _ = check_router(ih, wh, nh, xh, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
        assert near == 0
        ref = ffn_reference(cfg, xh, ih, wh, nh, rh)
        if cfg.x_dtype == "bf16":
            assert_close(yh, ref, BF16_RTOL, bf16_atol(ref), cfg.name)
        else:
            assert_close(yh, ref, F32_RTOL, f32_atol(ref), cfg.name)
    finally:
        layer.free()


def test_dense_projection_writes_only_inside_its_buffer(ctx):
    from int4_grouped_expert_router_gb300 import synth
    import oracle.moe as O
    for S, O_, I in ((1, 7000, 200), (3, 200, 7000)):
        p, sc = synth.expert_tensor(synth.stream_seed(31, O_, I), O_, I, 0)
        h = B.coli_expert_upload(ctx, torch.from_numpy(p), torch.from_numpy(sc), O_, I, 0)
        try:
            x = torch.from_numpy(synth.normal(synth.stream_seed(32, S), S * I).reshape(S, I)).cuda()
            by, y = guarded((S, O_), torch.float32)
            B.coli_w4_linear(ctx, h, x, None, y)
            assert B.coli_check_error(ctx) == 0
            assert intact(by, y.numel())
            ref = O.w4_linear(x.cpu().numpy(), O.Tensor(p, sc, O_, I, 0))
            assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), f"w4_linear S={S} O={O_} I={I}")
        finally:
            B.coli_expert_free(ctx, h)
