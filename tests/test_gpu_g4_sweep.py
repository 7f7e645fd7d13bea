"""Grouped-scale (g4) sweep: 50 random trials x 3 experts in one launch, as c/backend_cuda.cu commit history,
commit "The grouped MoE kernels were per-row-only", tests its g4 kernels: group size 64 with a tail group,
and a per-row member in the same launch. Every trial draws fresh experts (gs = 64, 0, 64), a fresh token, a
fresh order of the three slots and fresh weights; y must match the oracle element by element with zero
mismatches (rel 1e-4, absolute term in units of rms(y), see tests/test_tolerance.py).

Two shapes: D = 200, I = 136 (tail groups of 8 columns in both the gate/up rows and the down rows) takes
the two-kernel GEMV path; D = 1024, I = 208 (a 16-column tail in the down rows) takes the streaming path.
"""
import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from int4_grouped_expert_router_gb300.workload import DeviceLayer, LayerConfig
from gpu_util import F32_RTOL, Ctx, assert_close, f32_atol, ffn_reference, to_np

pytestmark = pytest.mark.gpu

TRIALS = 50


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


@pytest.mark.parametrize("D,I", [(200, 136), (1024, 208)], ids=["gemv-D200-I136", "stream-D1024-I208"])
def test_g4_sweep_50_trials_3_experts(ctx, D, I):
    worst = 0.0
    for trial in range(TRIALS):
        cfg = LayerConfig(f"g4-{trial}", D=D, I=I, E=3, K=3, gs="mixed:64",
                          seed=synth.stream_seed(synth.BASE_SEED, "g4 sweep", D, trial))
        layer = DeviceLayer(ctx, cfg)
        try:
            x = synth.normal(synth.stream_seed(cfg.seed, "x"), D).reshape(1, D)
            resid = synth.normal(synth.stream_seed(cfg.seed, "r"), D).reshape(1, D)
            order = synth.permutation(synth.stream_seed(cfg.seed, "order"), 3).astype(np.int32)
            w = synth.uniform(synth.stream_seed(cfg.seed, "w"), 3, 0.25, 1.25).astype(np.float32).reshape(1, 3)
            idx = order.reshape(1, 3)
            y = torch.empty(1, D, device="cuda")
            B.coli_expert_group(ctx, torch.from_numpy(x).cuda(), torch.from_numpy(idx).cuda(),
                                torch.from_numpy(w).cuda(), None, 3, torch.from_numpy(resid).cuda(), y)
            assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
            ref = ffn_reference(cfg, x, idx, w, None, resid)
            stats = assert_close(to_np(y), ref, F32_RTOL, f32_atol(ref), f"trial {trial}")
            assert stats["n_bad"] == 0
            worst = max(worst, stats["max_abs"] / f32_atol(ref))
        finally:
            layer.free()
    print(f"D={D} I={I}: {TRIALS} trials x 3 experts, worst |err| / abs term {worst:.3f}")
