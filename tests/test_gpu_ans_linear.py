"""The compressed tier's fused block decode + GEMV (coli_ans_w4_linear) against the oracle's w4_linear.

The tensor's packed bytes are uploaded as a compressed stream (coli_ans_upload) and y = resid + W x is
computed from the stream without writing the raw tensor: the expert shapes of the decode layer (gate/up
[2048 x 6144], down [6144 x 2048]), rows that straddle blocks irregularly (I = 1000: 500-byte rows) with a
64-column tail group, the smallest I (256) with fewer bytes than one block, bf16 activations with a
residual, and incompressible (uniform) nibbles. Results are bit-identical from call to call; shapes that
do not match the stream are rejected.
"""
import numpy as np
import pytest
import torch

import oracle.moe as O
from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from gpu_util import BF16_RTOL, F32_RTOL, Ctx, assert_close, bf16_atol, f32_atol, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


def make_tensor(seed, rows, cols, gs, kind="gauss"):
    nbytes = rows * cols // 2
    if kind == "gauss":
        packed = synth.gaussian_nibble_bytes(synth.stream_seed(seed, "ans-lin-w"), nbytes, 2.5)
    else:
        packed = synth.random_bytes(synth.stream_seed(seed, "ans-lin-w"), nbytes)
    ns = rows if gs == 0 else rows * ((cols + gs - 1) // gs)
    scales = synth.uniform(synth.stream_seed(seed, "ans-lin-s"), ns, 0.005, 0.02).astype(np.float32)
    return packed, scales


# (name, O, I, gs, activations, residual, nibbles)
CASES = [
    ("gate-2048x6144", 2048, 6144, 0, torch.float32, False, "gauss"),
    ("down-6144x2048", 6144, 2048, 0, torch.float32, True, "gauss"),
    ("I1000-g64-tail", 300, 1000, 64, torch.float32, True, "gauss"),
    ("I256-g32-small", 7, 256, 32, torch.float32, False, "gauss"),
    ("bf16-513x6144", 513, 6144, 0, torch.bfloat16, True, "gauss"),
    ("uniform-nibbles", 129, 2050, 0, torch.float32, False, "uniform"),
]


@pytest.mark.parametrize("name,Orows,I,gs,dt,with_resid,kind", CASES, ids=[c[0] for c in CASES])
def test_fused_decode_gemv_matches_oracle(ctx, name, Orows, I, gs, dt, with_resid, kind):
    packed, scales = make_tensor(len(name), Orows, I, gs, kind)
    h = B.coli_ans_upload(ctx, packed.tobytes())
    try:
        x = synth.normal(synth.stream_seed(7, name, "x"), I).astype(np.float32)
        resid = synth.normal(synth.stream_seed(7, name, "r"), Orows).astype(np.float32) if with_resid else None
        if dt == torch.bfloat16:
            x = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
            if resid is not None:
                resid = synth.bf16_bits_to_f32(synth.to_bf16_bits(resid))
        xt = torch.from_numpy(x).cuda().to(dt)
        rt = torch.from_numpy(resid).cuda().to(dt) if resid is not None else None
        st = torch.from_numpy(scales).cuda()
        y = torch.empty(Orows, dtype=dt, device="cuda")
        B.coli_ans_w4_linear(ctx, h, st, Orows, I, gs, xt, rt, y)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        ref = O.w4_linear(x, O.Tensor(packed, scales, Orows, I, gs), resid)[0]
        if dt == torch.bfloat16:
            assert_close(to_np(y), ref, BF16_RTOL, bf16_atol(ref), name)
        else:
            stats = assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), name)
            print(name, stats)
        y2 = torch.empty_like(y)
        B.coli_ans_w4_linear(ctx, h, st, Orows, I, gs, xt, rt, y2)
        assert torch.equal(y, y2)
    finally:
        B.coli_ans_free(ctx, h)


def test_shapes_that_do_not_match_the_stream_are_rejected(ctx):
    packed, scales = make_tensor(5, 64, 512, 0)
    h = B.coli_ans_upload(ctx, packed.tobytes())
    try:
        st = torch.from_numpy(scales).cuda()
        x = torch.zeros(512, device="cuda")
        y = torch.empty(64, device="cuda")
        for Orows, I, gs in ((64, 510, 0), (33, 1000, 0), (128, 250, 0), (64, 512, 3)):
            with pytest.raises((B.ColiError, ValueError)):
                B.coli_ans_w4_linear(ctx, h, st, Orows, I, gs, torch.zeros(I, device="cuda"),
                                     None, torch.empty(Orows, device="cuda"))
        B.coli_ans_w4_linear(ctx, h, st, 64, 512, 0, x, None, y)  # the matching shape works
        assert B.coli_check_error(ctx) == 0
    finally:
        B.coli_ans_free(ctx, h)
