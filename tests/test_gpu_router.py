"""Device router (logits GEMV, sigmoid, bias-augmented top-K, weights, top-p, norm, scale) vs the oracle."""
import numpy as np
import pytest
import torch

from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from gpu_util import Ctx, check_router

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


def run_router(ctx, x, Wr, bias, K, topp, norm, rs, dtype=torch.float32):
    S, E = x.shape[0], Wr.shape[0]
    xt = torch.from_numpy(x).cuda().to(dtype)
    idx = torch.full((S, K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((S, K), -7.0, dtype=torch.float32, device="cuda")
    n = torch.full((S,), -7, dtype=torch.int32, device="cuda")
    B.coli_router_select(ctx, xt, torch.from_numpy(Wr).cuda(), None if bias is None else torch.from_numpy(bias).cuda(),
                         K, topp, norm, rs, idx, w, n)
    assert B.coli_check_error(ctx) == 0
    return idx.cpu().numpy(), w.cpu().numpy(), n.cpu().numpy()


def test_tiny_config(ctx):
    x, Wr, bias = synth.router_inputs(synth.BASE_SEED, 1, 256, 16)
    idx, w, n = run_router(ctx, x, Wr, bias, 4, 0.0, True, 2.5)
    near, _ = check_router(idx, w, n, x, Wr, bias, 4, 0.0, True, 2.5)
    assert near == 0
    assert abs(float(w.sum()) - 2.5) < 1e-5


def test_random_trials_mixed_options(ctx):
    """200 random trials over E, K, S, top-p, norm_topk and routed_scale; near-ties counted."""
    near_total = 0
    for trial in range(200):
        E = [16, 64, 256, 100, 300][trial % 5]
        K = 1 + trial % 8
        S = 1 + trial % 3
        D = [256, 512, 6144, 200][trial % 4]
        topp = [0.0, 0.5, 0.7, 0.9, 1.0][trial % 5 if trial % 7 else 2]
        norm = trial % 3 != 0
        rs = [1.0, 2.5, 0.75][trial % 3]
        x, Wr, bias = synth.router_inputs(synth.stream_seed(synth.BASE_SEED, "router-trial", trial), S, D, E)
        idx, w, n = run_router(ctx, x, Wr, bias, K, topp, norm, rs)
        near, _ = check_router(idx, w, n, x, Wr, bias, K, topp, norm, rs)
        near_total += near
    print(f"router trials: 200, near-tie tokens: {near_total}")
    assert near_total <= 2


def test_exact_ties_go_to_lower_index(ctx):
    E, D, K = 64, 128, 8
    x = np.zeros((1, D), np.float32)
    x[0, 0] = 1.0
    Wr = np.zeros((E, D), np.float32)
    bias = (np.arange(E) % 4).astype(np.float32) * np.float32(0.125)   # many exact ties
    idx, w, n = run_router(ctx, x, Wr, bias, K, 0.0, True, 1.0)
    assert idx[0].tolist() == [3, 7, 11, 15, 19, 23, 27, 31]
    near, _ = check_router(idx, w, n, x, Wr, bias, K, 0.0, True, 1.0)
    assert near == 0


def test_no_bias_and_k_equals_e(ctx):
    x, Wr, _ = synth.router_inputs(5, 2, 96, 32)
    idx, w, n = run_router(ctx, x, Wr, None, 32, 0.0, False, 1.0)
    for t in range(2):
        assert sorted(idx[t].tolist()) == list(range(32))
    near, _ = check_router(idx, w, n, x, Wr, None, 32, 0.0, False, 1.0)
    assert near == 0


def test_bf16_activations(ctx):
    x, Wr, bias = synth.router_inputs(9, 4, 6144, 256, zipf=True)
    xb = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    idx, w, n = run_router(ctx, xb, Wr, bias, 8, 0.0, True, 2.5, dtype=torch.bfloat16)
    near, _ = check_router(idx, w, n, xb, Wr, bias, 8, 0.0, True, 2.5)
    assert near <= 1


def test_many_tokens(ctx):
    x, Wr, bias = synth.router_inputs(11, 70, 512, 256)
    idx, w, n = run_router(ctx, x, Wr, bias, 8, 0.9, True, 2.5)
    near, _ = check_router(idx, w, n, x, Wr, bias, 8, 0.9, True, 2.5)
    assert near <= 1


@pytest.mark.parametrize("E,K,S", [(1024, 8, 1), (1025, 32, 1), (1500, 8, 3), (4096, 32, 1), (4096, 8, 20), (2048, 16, 17)])
def test_expert_counts_up_to_the_limit(ctx, E, K, S):
    """E up to COLI_MAX_EXPERTS: more than 32 experts per selecting lane above E = 1024 (the decode
    router for S < 16, the batched router's selection kernel for S >= 16)."""
    assert E <= B.COLI_MAX_EXPERTS and K <= B.COLI_MAX_K
    x, Wr, bias = synth.router_inputs(synth.stream_seed(synth.BASE_SEED, "router-large-e", E * 100 + K), S, 256, E)
    idx, w, n = run_router(ctx, x, Wr, bias, K, 0.9 if S > 1 else 0.0, True, 2.5)
    near, _ = check_router(idx, w, n, x, Wr, bias, K, 0.9 if S > 1 else 0.0, True, 2.5)
    assert near <= 1
    assert (idx[:, 0] >= 1024).any() or E == 1024 or S == 1  # experts past the first 1024 do get chosen


def test_high_index_expert_wins(ctx):
    """The top expert is the last one of E = 4096: only a selection that sees every lane's 128
    experts finds it first."""
    E, D, K = 4096, 64, 4
    x = np.zeros((1, D), np.float32)
    x[0, 0] = 1.0
    Wr = np.zeros((E, D), np.float32)
    Wr[E - 1, 0] = 3.0
    Wr[E - 2, 0] = 2.0
    Wr[1500, 0] = 1.0
    Wr[7, 0] = 0.5
    idx, w, n = run_router(ctx, x, Wr, None, K, 0.0, False, 1.0)
    assert idx[0].tolist() == [E - 1, E - 2, 1500, 7]
    near, _ = check_router(idx, w, n, x, Wr, None, K, 0.0, False, 1.0)
    assert near == 0


@pytest.mark.parametrize("S", [15, 16, 65536])
def test_token_counts(ctx, S):
    """Both sides of the switch to the many-token router (S = 16), and S = COLI_MAX_TOKENS."""
    x, Wr, bias = synth.router_inputs(synth.stream_seed(synth.BASE_SEED, "router-tokens", S), S, 64, 16)
    idx, w, n = run_router(ctx, x, Wr, bias, 4, 0.8, True, 2.5)
    near, _ = check_router(idx, w, n, x, Wr, bias, 4, 0.8, True, 2.5)  # every other token exact
    print(f"S={S}: near-tie tokens {near}")
    assert near <= S // 1000 + 1


def test_nonfinite_activation_reported(ctx):
    x, Wr, bias = synth.router_inputs(12, 1, 128, 16)
    x[0, 5] = np.nan
    xt = torch.from_numpy(x).cuda()
    idx = torch.empty(1, 4, dtype=torch.int32, device="cuda")
    w = torch.empty(1, 4, dtype=torch.float32, device="cuda")
    B.coli_router_select(ctx, xt, torch.from_numpy(Wr).cuda(), torch.from_numpy(bias).cuda(), 4, 0.0, True, 1.0, idx, w)
    assert B.coli_check_error(ctx) == B.COLI_E_NONFINITE
    assert B.coli_check_error(ctx) == 0   # cleared


def test_argument_errors(ctx):
    x = torch.zeros(1, 64, device="cuda")
    Wr = torch.zeros(8, 64, device="cuda")
    idx = torch.empty(1, 9, dtype=torch.int32, device="cuda")
    w = torch.empty(1, 9, dtype=torch.float32, device="cuda")
    with pytest.raises(B.ColiError) as ei:
        B.coli_router_select(ctx, x, Wr, None, 9, 0.0, True, 1.0, idx, w)   # K > E
    assert ei.value.code == B.COLI_E_INVAL
