"""coli_router_select_noalloc: the router entry with fixed device scratch, against coli_router_select
and against the oracle.

Collected last (file name) so that it runs both alone and after every other GPU test; it creates
its own contexts and depends on no state left by other tests.
"""
import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from gpu_util import Ctx, check_router

pytestmark = pytest.mark.gpu

FIXED_CELLS = 65536  # S * E limit of the fixed scratch, as documented in the header


def _outputs(S, K):
    return (torch.full((S, K), -7, dtype=torch.int32, device="cuda"),
            torch.full((S, K), -7.0, dtype=torch.float32, device="cuda"),
            torch.full((S,), -7, dtype=torch.int32, device="cuda"))


def _inputs(seed, S, D, E, dtype=torch.float32, zipf=False):
    x, Wr, bias = synth.router_inputs(seed, S, D, E, zipf=zipf)
    return (torch.from_numpy(x).cuda().to(dtype), torch.from_numpy(Wr).cuda(), torch.from_numpy(bias).cuda())


CASES = [
    # (S, D, E, K, topp, norm_topk, routed_scale, dtype)
    (1, 6144, 256, 8, 0.0, True, 2.5, torch.float32),
    (4, 6144, 256, 8, 0.9, True, 2.5, torch.bfloat16),
    (3, 200, 100, 5, 0.7, False, 1.0, torch.float32),
    (256, 512, 256, 8, 0.0, True, 2.5, torch.float32),  # S * E exactly at the limit
    (1, 256, 4096, 32, 0.0, True, 2.5, torch.float32),   # more than 1024 experts: the large-E selection
    (16, 128, 4096, 8, 0.9, True, 2.5, torch.float32),   # ... in the many-token router, S * E at the limit
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c[0]}-D{c[1]}-E{c[2]}-K{c[3]}")
def test_matches_router_select_on_two_calls_in_a_row(case):
    S, D, E, K, topp, norm, rs, dtype = case
    c = Ctx()
    try:
        for call in range(2):  # the second call reuses the scratch the first one left behind
            x, Wr, bias = _inputs(synth.stream_seed(synth.BASE_SEED, "noalloc", S, E, call), S, D, E, dtype)
            ia, wa, na = _outputs(S, K)
            ib, wb, nb = _outputs(S, K)
            B.coli_router_select_noalloc(c.ctx, x, Wr, bias, K, topp, norm, rs, ia, wa, na)
            B.coli_router_select(c.ctx, x, Wr, bias, K, topp, norm, rs, ib, wb, nb)
            assert B.coli_check_error(c.ctx) == 0
            assert torch.equal(ia, ib), call
            assert torch.equal(na, nb), call
            assert np.array_equal(wa.cpu().numpy().view(np.uint32), wb.cpu().numpy().view(np.uint32)), call
            assert (ia >= 0).any()
            # and against the oracle directly (exact indices except near-ties, weights rel 1e-4 / abs 1e-5)
            xh = x.float().cpu().numpy().astype(np.float64)
            near, _ = check_router(ia.cpu().numpy(), wa.cpu().numpy(), na.cpu().numpy(), xh, Wr.cpu().numpy(),
                                   bias.cpu().numpy(), K, topp, norm, rs)
            assert near <= max(1, S // 64), near
    finally:
        c.close()


@pytest.mark.parametrize("S", [1, 16], ids=["decode-path", "many-token-path"])
def test_device_memory_unchanged_by_calls(S):
    """After a warm-up call (which looks up the scratch address), calls leave free memory as it was:
    S = 1 takes the one-kernel router (its launch counter only grows), S = 16 the many-token
    router (three kernels)."""
    D, E, K = 2048, 256, 8
    c = Ctx()
    try:
        x, Wr, bias = _inputs(3, S, D, E)
        idx, w, n = _outputs(S, K)
        B.coli_router_select_noalloc(c.ctx, x, Wr, bias, K, 0.0, True, 2.5, idx, w, n)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for _ in range(3):
            B.coli_router_select_noalloc(c.ctx, x, Wr, bias, K, 0.0, True, 2.5, idx, w, n)
        assert B.coli_check_error(c.ctx) == 0
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0
    finally:
        c.close()


def test_sizes_over_the_limit_rejected():
    E, K, D = 256, 8, 64
    S = FIXED_CELLS // E + 1
    c = Ctx()
    try:
        x = torch.zeros(S, D, device="cuda")
        Wr = torch.zeros(E, D, device="cuda")
        idx, w, n = _outputs(S, K)
        with pytest.raises(B.ColiError) as ei:
            B.coli_router_select_noalloc(c.ctx, x, Wr, None, K, 0.0, True, 1.0, idx, w, n)
        assert ei.value.code == B.COLI_E_INVAL
        assert "limit" in B.coli_last_error(c.ctx)
        assert (idx == -7).all()  # nothing was launched
        assert B.coli_check_error(c.ctx) == 0
    finally:
        c.close()
