"""The dense int4 projection (coli_w4_linear) and a layer with a shared expert, against the oracle.

- coli_w4_linear over every scale layout (per row, chunk groups with a tail, generic even gs), ragged
  widths, f32 and bf16, with and without a residual, one token (the down kernel's TMA rings) and many
  (several finishing segments per CTA and token switches inside a segment), at the widest blocks and
  at 6144 x 6144.
- y written in place over the residual; argument errors leave the context usable.
- The shared expert, commit "CUDA batch MLA attention, ..., W4A16 kernels": an always-chosen expert
  of weight 1, registered outside the router's ids. Two ways: the router appends it after each
  token's kept slots (coli_router_select_shared, checked slot for slot against the oracle's
  append_shared of the plain router's output) and one coli_expert_group call runs K + 1 slots; or
  it is issued as its own group next to the routed group ([resid] issue/take). Both against the
  oracle's routed + shared block.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.moe as O
from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, host_expert, router_host_inputs
from gpu_util import BF16_RTOL, F32_RTOL, Ctx, assert_close, bf16_atol, f32_atol, oracle_experts, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


def make_case(seed, O_, I_, gs, S, dtype):
    p, s = synth.expert_tensor(synth.stream_seed(seed, "W"), O_, I_, gs)
    x = synth.normal(synth.stream_seed(seed, "x"), S * I_).reshape(S, I_)
    r = synth.normal(synth.stream_seed(seed, "r"), S * O_).reshape(S, O_)
    if dtype == "bf16":
        x = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
        r = synth.bf16_bits_to_f32(synth.to_bf16_bits(r))
    return O.Tensor(p, s, O_, I_, gs), x, r


def dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


CASES = [
    # name, O, I, gs, S, dtype, residual
    ("tiny-row", 64, 128, 0, 1, "f32", True),
    ("ragged-g64-tail", 203, 200, 64, 3, "f32", False),
    ("generic-gs6-bf16", 50, 96, 6, 2, "bf16", True),
    ("g32", 1000, 1024, 32, 5, "f32", True),
    ("tokens-g64-bf16", 256, 512, 64, 64, "bf16", True),
    ("segments", 4096, 256, 0, 64, "f32", True),
    ("wide-1024-threads", 96, 20000, 128, 2, "f32", True),
    ("square-6144", 6144, 6144, 0, 1, "f32", True),
    # one token runs on the down kernel's TMA rings: every scale layout, bf16 activations, wide rows
    ("s1-generic-gs6-bf16", 50, 96, 6, 1, "bf16", True),
    ("s1-g64-tail-bf16", 203, 200, 64, 1, "bf16", False),
    ("s1-g32-f32", 1000, 1000, 32, 1, "f32", True),
    ("s1-wide-640-threads", 96, 20000, 128, 1, "f32", True),
    ("s1-bf16-6144", 6144, 6144, 0, 1, "bf16", True),
    # one token through tensors the streaming kernel takes (I a multiple of 1024 up to 6144, O of 16, gs 0 or 32 k)
    ("s1-stream-g64", 2048, 6144, 64, 1, "f32", True),
    ("s1-stream-g32-bf16", 4096, 2048, 32, 1, "bf16", False),
    ("s1-stream-3-units", 48, 1024, 0, 1, "f32", True),
    ("s1-stream-I5120", 1040, 5120, 0, 1, "f32", False),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_linear_matches_oracle(ctx, case):
    name, O_, I_, gs, S, dtype, with_resid = case
    T, x, r = make_case(sum(map(ord, name)), O_, I_, gs, S, dtype)
    h = B.coli_expert_upload(ctx, torch.from_numpy(T.packed.reshape(-1).copy()), torch.from_numpy(T.scales.copy()),
                             O_, I_, gs)
    try:
        assert B.coli_tensor_shape(ctx, h) == (O_, I_, gs)
        xt = dev(x, dtype)
        rt = dev(r, dtype) if with_resid else None
        y = torch.full((S, O_), 7.0, device="cuda", dtype=xt.dtype)
        B.coli_w4_linear(ctx, h, xt, rt, y)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        ref = O.w4_linear(to_np(xt), T, to_np(rt) if with_resid else None)
        rtol, atol = (BF16_RTOL, bf16_atol(ref)) if dtype == "bf16" else (F32_RTOL, f32_atol(ref))
        print(name, assert_close(to_np(y), ref, rtol, atol, name))
        y2 = torch.empty_like(y)
        B.coli_w4_linear(ctx, h, xt, rt, y2)
        assert torch.equal(y, y2)  # run to run
    finally:
        B.coli_expert_free(ctx, h)


def test_linear_in_place_and_errors(ctx):
    T, x, r = make_case(5, 300, 160, 32, 4, "f32")
    h = B.coli_expert_upload(ctx, torch.from_numpy(T.packed.reshape(-1).copy()), torch.from_numpy(T.scales.copy()),
                             300, 160, 32)
    try:
        xt, rt = dev(x, "f32"), dev(r, "f32")
        y = torch.empty(4, 300, device="cuda")
        B.coli_w4_linear(ctx, h, xt, rt, y)
        B.coli_w4_linear(ctx, h, xt, rt, rt)  # y = resid: in place
        assert B.coli_check_error(ctx) == 0
        assert torch.equal(y, rt)
        lib = B.library()
        p = ctypes.c_void_p(xt.data_ptr())
        assert lib.coli_w4_linear(ctx, h + 1000, p, B.COLI_DTYPE_F32, 4, None, p) == B.COLI_E_INVAL
        assert lib.coli_w4_linear(ctx, h, p, B.COLI_DTYPE_F32, 0, None, p) == B.COLI_E_INVAL
        assert lib.coli_w4_linear(ctx, h, p, 7, 4, None, p) == B.COLI_E_INVAL
        assert lib.coli_w4_linear(ctx, h, None, B.COLI_DTYPE_F32, 4, None, p) == B.COLI_E_INVAL
        B.coli_profile_enable(ctx, 1)
        B.coli_profile_read(ctx, B.COLI_KERNEL_LINEAR)
        B.coli_w4_linear(ctx, h, xt, None, y)
        assert B.coli_profile_read(ctx, B.COLI_KERNEL_LINEAR)[1] == 1
        B.coli_profile_enable(ctx, 0)
        assert B.coli_check_error(ctx) == 0
        ref = O.w4_linear(x, T)
        assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), "after errors")
    finally:
        B.coli_expert_free(ctx, h)


@pytest.mark.parametrize("cfg", [
    LayerConfig("shared-S1", D=512, I=256, E=16, K=4, routed_scale=2.5),
    LayerConfig("shared-S4-g64-bf16", D=512, I=320, E=16, K=4, S=4, gs=64, topp=0.9, x_dtype="bf16"),
    # 32 tokens x 5 slots over 16 experts: the batched router and the tensor-core expert path
    LayerConfig("shared-S32-tc", D=256, I=128, E=16, K=4, S=32, gs=64, x_dtype="bf16", zipf=True, topp=0.8),
], ids=lambda c: c.name)
def test_shared_expert_layer(ctx, cfg):
    layer = DeviceLayer(ctx, cfg)
    e_sh = cfg.E  # outside the router's ids 0..E-1
    hs = []
    try:
        for (p, s, rows, cols, gs) in host_expert(cfg, e_sh):
            hs.append(B.coli_expert_upload(ctx, torch.from_numpy(p.reshape(-1).copy()), torch.from_numpy(s.copy()),
                                           rows, cols, gs))
        B.coli_expert_table_set(ctx, e_sh, *hs)
        x, Wr, bias, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        r = layer.outputs()
        B.coli_router_select(ctx, xt, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale,
                             r["idx"], r["w"], r["n_sel"])
        sh_idx = torch.full((cfg.S, 1), e_sh, dtype=torch.int32, device="cuda")
        sh_w = torch.ones(cfg.S, 1, device="cuda")
        assert B.coli_expert_group_issue(ctx, xt, r["idx"], r["w"], r["n_sel"], cfg.K) == 0
        assert B.coli_expert_group_issue(ctx, xt, sh_idx, sh_w, None, 1) == 1
        y = torch.empty_like(xt)
        B.coli_expert_group_take(ctx, rt, y)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        idx, w, n = (to_np(r[k]) for k in ("idx", "w", "n_sel"))
        xw, rw = to_np(xt), to_np(rt)
        experts = oracle_experts(cfg, idx)
        shared = oracle_experts(cfg, [e_sh])[e_sh]
        ref = O.moe_block_with_shared(xw, experts, idx, w, n, shared, rw)
        rtol, atol = (BF16_RTOL, bf16_atol(ref)) if cfg.x_dtype == "bf16" else (F32_RTOL, f32_atol(ref))
        if cfg.name.endswith("-tc"):  # groups with many rows per expert may run on the tensor cores
            from test_gpu_prefill import TC_RTOL, tc_atol
            rtol, atol = TC_RTOL, tc_atol(ref)
        print(cfg.name, assert_close(to_np(y), ref, rtol, atol, cfg.name))
        # the router appends the shared slot; one grouped call with K + 1 slots
        i2 = torch.empty(cfg.S, cfg.K + 1, dtype=torch.int32, device="cuda")
        w2 = torch.empty(cfg.S, cfg.K + 1, device="cuda")
        n2 = torch.empty(cfg.S, dtype=torch.int32, device="cuda")
        B.coli_router_select_shared(ctx, xt, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale,
                                    e_sh, i2, w2, n2)
        ia, wa, na = O.append_shared(idx, w, n, e_sh)
        assert np.array_equal(to_np(i2), ia) and np.array_equal(to_np(w2), wa) and np.array_equal(to_np(n2), na)
        y2 = torch.empty_like(xt)
        B.coli_expert_group(ctx, xt, i2, w2, n2, cfg.K + 1, rt, y2)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        print(cfg.name, "one call", assert_close(to_np(y2), ref, rtol, atol, cfg.name + " one call"))
    finally:
        B.coli_expert_table_set(ctx, e_sh, 0, 0, 0)
        for h in hs:
            B.coli_expert_free(ctx, h)
        layer.free()


@pytest.mark.parametrize("O_,I_,gs", [(6144, 6144, 0), (2048, 6144, 64)])
def test_one_token_streaming_matches_the_ring_form(O_, I_, gs):
    """One token: the streaming kernel (default) against the down-kernel ring form (COLI_DECODE_STREAM=0)."""
    from gpu_util import Ctx
    T, x, r = make_case(O_ + gs, O_, I_, gs, 1, "f32")
    cs, c2 = Ctx(), Ctx.with_env(COLI_DECODE_STREAM=0)
    hs = [B.coli_expert_upload(c.ctx, torch.from_numpy(T.packed.reshape(-1).copy()), torch.from_numpy(T.scales.copy()),
                               O_, I_, gs) for c in (cs, c2)]
    try:
        xt, rt = dev(x, "f32"), dev(r, "f32")
        ys = [torch.empty(1, O_, device="cuda") for _ in range(2)]
        for c, h, y in zip((cs, c2), hs, ys):
            B.coli_profile_enable(c.ctx, 1)
            B.coli_profile_read(c.ctx, B.COLI_KERNEL_LINEAR)
            B.coli_w4_linear(c.ctx, h, xt, rt, y)
            assert B.coli_check_error(c.ctx) == 0, B.coli_last_error(c.ctx)
            assert B.coli_profile_read(c.ctx, B.COLI_KERNEL_LINEAR)[1] == 1
        ref = O.w4_linear(x, T, r)
        assert_close(to_np(ys[0]), ref, F32_RTOL, f32_atol(ref), "streaming")
        assert_close(to_np(ys[1]), to_np(ys[0]), 2 * F32_RTOL, 2 * f32_atol(ref), "streaming vs rings")
    finally:
        for c, h in zip((cs, c2), hs):
            B.coli_expert_free(c.ctx, h)
            c.close()
