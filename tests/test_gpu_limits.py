"""The grouped expert FFN at the header's size limits, against the oracle.

- D = COLI_MAX_GROUP_DIM (8192): eight warps per gate/up CTA, one CTA per SM.
- D = 7000 (ragged, 219 column chunks) with 64-column groups and a 24-column tail group.
- I = 32768 (COLI_MAX_DIM): 1024 threads per down row, the route-parallel down kernel.
- S = COLI_MAX_GROUP_TOKENS (1024) tokens on the GEMV path.
- K = E = 32 (COLI_MAX_K): every expert chosen by every token.
- Down kernels whose block (K ceil(I/1024) 32 threads) is smaller than a 64-row segment or its row-scale cells,
  and blocks of 576 and 768 threads (9 and 12 slots).
- bf16 rows that are not 16-byte aligned, and the tensor-core path at D = 8192 (checked with its tolerance).
"""
import pytest

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig, router_host_inputs
from gpu_util import BF16_RTOL, F32_RTOL, Ctx, assert_close, bf16_atol, check_router, f32_atol, ffn_reference, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


LIMITS = [
    LayerConfig("D8192-f32", D=8192, I=128, E=8, K=4),
    LayerConfig("D8192-S2-bf16", D=8192, I=128, E=8, K=4, S=2, x_dtype="bf16"),
    LayerConfig("D7000-g64-tail", D=7000, I=200, E=8, K=3, gs=64),
    LayerConfig("I32768", D=64, I=32768, E=4, K=2),
    LayerConfig("S1024", D=128, I=64, E=16, K=8, S=1024, topp=0.9),
    LayerConfig("K32-E32", D=128, I=64, E=32, K=32, S=2, gs="mixed:32"),
    # one slot of 32 threads per down row range of 40 rows, and 4 slots of 32 threads for 54 rows: the down
    # kernel's block is smaller than a segment's rows (and its row-scale cells)
    LayerConfig("K1-D6144-I128", D=6144, I=128, E=4, K=1),
    LayerConfig("K4-D6144-I1024", D=6144, I=1024, E=8, K=4, gs="mixed:64"),
    # 9 and 12 slots of 64 threads: the 640- and 768-thread down kernels (a shared expert after 8 or 11 routed)
    LayerConfig("K9-I2048", D=256, I=2048, E=16, K=9),
    LayerConfig("K12-I2048", D=320, I=2048, E=16, K=12, gs="mixed:64"),
    # bf16 rows of 200 columns (400 bytes: not 16-byte aligned after row 0), one and several tokens
    LayerConfig("bf16-D200-S1", D=200, I=136, E=12, K=3, x_dtype="bf16"),
    LayerConfig("bf16-D200-S3", D=200, I=136, E=12, K=3, S=3, x_dtype="bf16"),
    # the tensor-core path at D = 8192: 128 K tiles of gate/up, 64 row tiles of down
    LayerConfig("tc-D8192", D=8192, I=256, E=8, K=4, S=64, gs=64, x_dtype="bf16", zipf=True),
]


@pytest.mark.parametrize("cfg", LIMITS, ids=lambda c: c.name)
def test_limits_match_oracle(ctx, cfg):
    assert cfg.D <= 8192 and cfg.I <= 32768 and cfg.S <= 1024 and cfg.K <= B.COLI_MAX_K
    layer = DeviceLayer(ctx, cfg)
    try:
        x, Wr, bias, resid = router_host_inputs(cfg)
        out = layer.outputs()
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        layer.step(xt, rt, out)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        idx, w, n, y = (to_np(out[k]) for k in ("idx", "w", "n_sel", "y"))
        xw, rw = to_np(xt), to_np(rt)
        near, _ = check_router(idx, w, n, xw, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
        assert near <= 1
        ref = ffn_reference(cfg, xw, idx, w, n, rw)
        if cfg.name.startswith("tc-"):
            from test_gpu_prefill import TC_NORM, TC_RTOL, tc_atol
            stats = assert_close(y, ref, TC_RTOL, tc_atol(ref), cfg.name)
            assert stats["norm_rel"] < TC_NORM, stats
        else:
            rtol, atol = (BF16_RTOL, bf16_atol(ref)) if cfg.x_dtype == "bf16" else (F32_RTOL, f32_atol(ref))
            stats = assert_close(y, ref, rtol, atol, cfg.name)
        print(cfg.name, stats)
    finally:
        layer.free()


@pytest.mark.parametrize("cfg", [
    LayerConfig("drop-all-S3", D=256, I=128, E=16, K=4, S=3),
    LayerConfig("drop-all-tc-S64", D=256, I=128, E=16, K=4, S=64, gs=64, x_dtype="bf16"),
], ids=lambda c: c.name)
def test_every_slot_dropped_gives_the_residual(ctx, cfg):
    """n_sel = 0 for every token: no route is kept, y = resid exactly (GEMV and tensor-core paths)."""
    import torch
    layer = DeviceLayer(ctx, cfg)
    try:
        x, _, _, resid = router_host_inputs(cfg)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        idx = torch.randint(0, cfg.E, (cfg.S, cfg.K), dtype=torch.int32, device="cuda")
        w = torch.rand(cfg.S, cfg.K, device="cuda")
        n = torch.zeros(cfg.S, dtype=torch.int32, device="cuda")
        y = torch.full_like(xt, 7.0)
        B.coli_expert_group(ctx, xt, idx, w, n, cfg.K, rt, y)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        assert torch.equal(y, rt)
        y0 = torch.full_like(xt, 7.0)
        B.coli_expert_group(ctx, xt, idx, w, n, cfg.K, None, y0)  # no residual: zeros
        assert B.coli_check_error(ctx) == 0
        assert not y0.abs().sum().item()
    finally:
        layer.free()
