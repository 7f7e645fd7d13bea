"""The one-launch router (fewer than 16 tokens, E <= 1024) against the oracle for every shape of its
grid: R logit rows per CTA (1, 2, 4, 8) times P column parts of D (1 to 4, as many as the selection
holds), over f32 and bf16 activations, D off the 4-column grid (element loads), ragged row blocks
(E % R != 0) and ragged parts (D % P != 0); the launch tags (words left by an earlier launch, with
more experts or another part count, are never taken for this launch's); and its bounded wait.
"""
import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from gpu_util import Ctx, check_router

pytestmark = pytest.mark.gpu


def route(ctx, x, Wr, bias, K, topp=0.0, norm=True, rs=2.5, dtype=torch.float32, check=True):
    S, E = x.shape[0], Wr.shape[0]
    xt = torch.from_numpy(x).cuda().to(dtype)
    idx = torch.full((S, K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((S, K), -7.0, dtype=torch.float32, device="cuda")
    n = torch.full((S,), -7, dtype=torch.int32, device="cuda")
    B.coli_router_select(ctx, xt, torch.from_numpy(Wr).cuda(), None if bias is None else torch.from_numpy(bias).cuda(),
                         K, topp, norm, rs, idx, w, n)
    if check:
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    return idx.cpu().numpy(), w.cpu().numpy(), n.cpu().numpy()


# (name, S, D, E, K, top-p, activations)
SHAPES = [
    ("S1-D6144-E256-K8", 1, 6144, 256, 8, 0.0, torch.float32),
    ("S4-D6144-E256-K8-bf16", 4, 6144, 256, 8, 0.9, torch.bfloat16),
    ("S3-D1000-E100-K6-topp", 3, 1000, 100, 6, 0.7, torch.float32),
    ("S2-D999-E60-K5-elementwise", 2, 999, 60, 5, 0.0, torch.float32),
    ("S1-D512-E1024-K16", 1, 512, 1024, 16, 0.0, torch.float32),
    ("S15-D64-E33-K32", 15, 64, 33, 32, 0.8, torch.float32),
    ("S1-D2050-E7-K7-bf16-odd", 1, 2050, 7, 7, 0.0, torch.bfloat16),
]


@pytest.mark.parametrize("rows,parts", [(1, 1), (2, 2), (4, 4), (8, 3), (4, 1), (1, 4)])
def test_every_grid_shape_matches_oracle(rows, parts):
    c = Ctx.with_env(COLI_ROUTER_ROWS=rows, COLI_ROUTER_PARTS=parts)
    try:
        for name, S, D, E, K, topp, dt in SHAPES:
            x, Wr, bias = synth.router_inputs(synth.stream_seed(synth.BASE_SEED, "router-grid", name), S, D, E)
            if dt == torch.bfloat16:
                x = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
            idx, w, n = route(c.ctx, x, Wr, bias, K, topp, dtype=dt)
            near, _ = check_router(idx, w, n, x, Wr, bias, K, topp, True, 2.5)
            assert near <= 1, (name, rows, parts)
            # bit-identical on repeat (the tags change, the result does not)
            idx2, w2, n2 = route(c.ctx, x, Wr, bias, K, topp, dtype=dt)
            assert np.array_equal(idx, idx2) and np.array_equal(w, w2) and np.array_equal(n, n2), name
    finally:
        c.close()


def test_words_of_earlier_launches_are_never_taken():
    """E = 256 with one token's inputs, then E = 64 and E = 256 with others: the second E = 256 launch
    finds its words' slots holding the first launch's values (same expert positions, older tags) and
    must wait for its own. Every launch matches the oracle, also with a different part count."""
    for parts in (1, 4):
        c = Ctx.with_env(COLI_ROUTER_PARTS=parts)
        try:
            for i, E in enumerate((256, 64, 256, 256, 8, 256)):
                x, Wr, bias = synth.router_inputs(synth.stream_seed(synth.BASE_SEED, "router-stale", parts, i), 2, 768, E)
                idx, w, n = route(c.ctx, x, Wr, bias, 8)
                near, _ = check_router(idx, w, n, x, Wr, bias, 8, 0.0, True, 2.5)
                assert near == 0, (parts, i, E)
        finally:
            c.close()


def test_exact_ties_across_and_within_lanes():
    """Equal choice scores everywhere (zero logits, a bias of four levels): the winners are the
    lowest indices of the top level, in index order, whatever the grid shape."""
    E, D, K = 256, 128, 16
    x = np.zeros((1, D), np.float32)
    x[0, 0] = 1.0
    Wr = np.zeros((E, D), np.float32)
    bias = (np.arange(E) % 4).astype(np.float32) * np.float32(0.125)
    for rows, parts in ((1, 1), (4, 4)):
        c = Ctx.with_env(COLI_ROUTER_ROWS=rows, COLI_ROUTER_PARTS=parts)
        try:
            idx, w, n = route(c.ctx, x, Wr, bias, K, 0.0, True, 1.0)
            assert idx[0].tolist() == list(range(3, 3 + 4 * K, 4))
            assert np.allclose(w[0], 1.0 / K)
        finally:
            c.close()


def test_bounded_wait_gives_up_then_healthy():
    """The last CTA withholds token 0's partial logits for one launch (test hook): the selection's wait
    gives up after the shortened limit, the call reports COLI_E_TIMEOUT and token 0 gets an empty route
    while token 1 is routed; the next call is healthy and matches the oracle. Nothing traps."""
    c = Ctx.with_env(COLI_TEST_WAIT_NS=20_000_000, COLI_TEST_WITHHOLD_ROUTER=1)
    try:
        x, Wr, bias = synth.router_inputs(synth.stream_seed(synth.BASE_SEED, "router-timeout"), 2, 1024, 64)
        idx, w, n = route(c.ctx, x, Wr, bias, 8, check=False)
        assert B.coli_check_error(c.ctx) == B.COLI_E_TIMEOUT
        assert n[0] == 0 and (idx[0] == -1).all() and (w[0] == 0).all()
        near, _ = check_router(idx[1:], w[1:], n[1:], x[1:], Wr, bias, 8, 0.0, True, 2.5)
        assert near == 0
        idx, w, n = route(c.ctx, x, Wr, bias, 8)
        near, _ = check_router(idx, w, n, x, Wr, bias, 8, 0.0, True, 2.5)
        assert near == 0
    finally:
        c.close()
