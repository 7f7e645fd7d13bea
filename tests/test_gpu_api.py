"""Behaviour of the boundary on a GPU: copy-on-upload, format checks, table rules, error consumption,
the COLI_FAIL_AFTER hook, and a healthy call after a failed allocation."""
import os

import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import F32_ATOL, F32_RTOL, Ctx, f32_atol, assert_close, ffn_reference, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture()
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


def upload_np(ctx, p, s, O, I, gs):
    return B.coli_expert_upload(ctx, torch.from_numpy(p), torch.from_numpy(s), O, I, gs)


def test_upload_copies_host_data(ctx):
    """The library keeps its own copy: scribbling and freeing the host buffers changes nothing."""
    cfg = LayerConfig("copy", D=128, I=64, E=2, K=2)
    x, _, _, _ = router_host_inputs(cfg)
    hs = {}
    for e in range(2):
        trip = []
        for which, (r, c) in (("gate", (64, 128)), ("up", (64, 128)), ("down", (128, 64))):
            p, s = synth.expert_tensor(synth.stream_seed(cfg.seed, "expert", e, which), r, c, 0)
            p2, s2 = p.copy(), s.copy()
            trip.append(upload_np(ctx, p2, s2, r, c, 0))
            p2[:] = 0xFF
            s2[:] = np.nan
            del p2, s2
        B.coli_expert_table_set(ctx, e, *trip)
        hs[e] = trip
    idx = np.array([[1, 0]], np.int32)
    w = np.array([[0.5, 2.0]], np.float32)
    outs = []
    for _ in range(64):   # sustained reuse of the device copies
        y = torch.empty(1, 128, device="cuda")
        B.coli_expert_group(ctx, torch.from_numpy(x).cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                            None, 2, None, y)
        outs.append(y)
    assert B.coli_check_error(ctx) == 0
    from workload_helpers import oracle_for_layer_seed
    ref = oracle_for_layer_seed(cfg, x, idx, w)
    for y in outs:
        assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), "after host scribble")


def test_upload_from_device_memory(ctx):
    p, s = synth.expert_tensor(77, 64, 96, 32)
    h = B.coli_expert_upload(ctx, torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda(), 64, 96, 32)
    assert h > 0
    B.coli_expert_free(ctx, h)


@pytest.mark.parametrize("O,I,gs", [(8, 7, 0), (8, 64, 3), (8, 64, -2)])
def test_upload_rejects_bad_formats(ctx, O, I, gs):
    p = np.zeros(O * ((I + 1) // 2), np.uint8)
    s = np.zeros(O if gs <= 0 else O * (-(-I // gs)), np.float32)
    h = B.library().coli_expert_upload(ctx, B._ptr(torch.from_numpy(p)), B._ptr(torch.from_numpy(s)), O, I, gs)
    assert h == 0
    assert B.coli_last_code(ctx) in (B.COLI_E_FORMAT, B.COLI_E_INVAL)
    # a failed upload leaves no pending runtime error: a normal upload works right after
    p2, s2 = synth.expert_tensor(1, 8, 64, 0)
    assert upload_np(ctx, p2, s2, 8, 64, 0) > 0


def test_table_shape_rules(ctx):
    mk = lambda O, I: upload_np(ctx, *synth.expert_tensor(O * 1000 + I, O, I, 0), O, I, 0)
    g, u, d = mk(32, 64), mk(32, 64), mk(64, 32)
    B.coli_expert_table_set(ctx, 3, g, u, d)
    with pytest.raises(B.ColiError) as ei:
        B.coli_expert_table_set(ctx, 4, g, u, mk(64, 30))   # down not [D x I]
    assert ei.value.code == B.COLI_E_FORMAT
    g2, u2, d2 = mk(16, 64), mk(16, 64), mk(64, 16)
    with pytest.raises(B.ColiError) as ei:
        B.coli_expert_table_set(ctx, 5, g2, u2, d2)          # different I from entry 3
    assert ei.value.code == B.COLI_E_FORMAT
    with pytest.raises(B.ColiError):
        B.coli_expert_free(ctx, g)                           # still referenced
    B.coli_expert_table_set(ctx, 3, 0, 0, 0)
    B.coli_expert_free(ctx, g)
    B.coli_expert_table_set(ctx, 5, g2, u2, d2)             # table empty again: new shape accepted
    with pytest.raises(B.ColiError):
        B.coli_expert_free(ctx, 999)


def test_fail_after_hook():
    os.environ["COLI_FAIL_AFTER"] = "2"
    try:
        c = Ctx()
    finally:
        del os.environ["COLI_FAIL_AFTER"]
    try:
        x, Wr, bias = synth.router_inputs(1, 1, 64, 8)
        args = (torch.from_numpy(x).cuda(), torch.from_numpy(Wr).cuda(), torch.from_numpy(bias).cuda(), 2, 0.0, True, 1.0,
                torch.empty(1, 2, dtype=torch.int32, device="cuda"), torch.empty(1, 2, device="cuda"))
        B.coli_router_select(c.ctx, *args)
        B.coli_router_select(c.ctx, *args)
        with pytest.raises(B.ColiError) as ei:
            B.coli_router_select(c.ctx, *args)
        assert ei.value.code == B.COLI_E_INJECTED
        # uploads are never gated
        assert upload_np(c.ctx, *synth.expert_tensor(2, 8, 16, 0), 8, 16, 0) > 0
    finally:
        c.close()
    # unset: no effect
    c2 = Ctx()
    try:
        x, Wr, bias = synth.router_inputs(1, 1, 64, 8)
        for _ in range(5):
            B.coli_router_select(c2.ctx, torch.from_numpy(x).cuda(), torch.from_numpy(Wr).cuda(), None, 2, 0.0, True, 1.0,
                                 torch.empty(1, 2, dtype=torch.int32, device="cuda"), torch.empty(1, 2, device="cuda"))
    finally:
        c2.close()


def test_healthy_call_after_failed_allocation(ctx):
    with pytest.raises(B.ColiError) as ei:
        B.coli_reserve(ctx, 65536, 4096, 32, 32768, 32768)   # far beyond device memory
    assert ei.value.code == B.COLI_E_OOM
    cfg = LayerConfig("after-oom", D=128, I=64, E=4, K=2)
    layer = DeviceLayer(ctx, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg)
        out = layer.outputs()
        layer.step(layer.act_tensor(x), layer.act_tensor(resid), out)
        assert B.coli_check_error(ctx) == 0
        ref = ffn_reference(cfg, x, to_np(out["idx"]), to_np(out["w"]), to_np(out["n_sel"]), resid)
        assert_close(to_np(out["y"]), ref, F32_RTOL, f32_atol(ref), "after failed alloc")
    finally:
        layer.free()
