"""Shared helpers of the GPU parity tests: library context, oracle comparison, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle.moe as O
from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from int4_grouped_expert_router_gb300.workload import host_expert

# Tolerances, elementwise |gpu - oracle| <= atol + rtol * |oracle|: rel 1e-4 / abs 1e-5 for f32
# activations and rel 1e-2 for bf16. The absolute term is stated for unit-scale outputs, so it is
# applied in units of the output's RMS magnitude when that exceeds 1 (an f32 evaluation's error
# at a cancellation point scales with the size of the terms, not with the tiny result).
F32_RTOL, F32_ATOL = 1e-4, 1e-5
BF16_RTOL = 1e-2
NEAR_TIE = 1e-6


def f32_atol(ref):
    ref = np.asarray(ref, np.float64)
    return F32_ATOL * max(1.0, float(np.sqrt(np.mean(ref * ref))))


def bf16_atol(ref):
    ref = np.asarray(ref, np.float64)
    return BF16_RTOL * 1e-2 * max(1.0, float(np.sqrt(np.mean(ref * ref))))


def oracle_experts(cfg, ids):
    out = {}
    for e in sorted(set(int(i) for i in np.asarray(ids).reshape(-1) if i >= 0)):
        g, u, d = host_expert(cfg, e)
        out[e] = tuple(O.Tensor(p, s, r, c, gs) for (p, s, r, c, gs) in (g, u, d))
    return out


def to_np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def check_router(idx_g, w_g, nsel_g, x, Wr, bias, K, topp, norm_topk, routed_scale):
    """Exact indices except near-ties (< 1e-6 apart in the oracle's choice score), counted.

    Returns (n_near_tie_tokens, max_weight_abs_err). Weights are compared (rel 1e-4 / abs 1e-5)
    whenever the indices agree.
    """
    idx_o, w_o, n_o, (z, s, c) = O.router_select(x, Wr, bias, K, topp, norm_topk, routed_scale)
    idx_g, w_g, nsel_g = np.asarray(idx_g), np.asarray(w_g), np.asarray(nsel_g)
    near, werr = 0, 0.0
    for t in range(x.shape[0]):
        if np.array_equal(idx_g[t], idx_o[t]) and nsel_g[t] == n_o[t]:
            err = np.abs(w_g[t].astype(np.float64) - w_o[t].astype(np.float64))
            assert np.all(err <= F32_ATOL + F32_RTOL * np.abs(w_o[t])), (t, w_g[t], w_o[t])
            werr = max(werr, float(err.max()))
            continue
        # a mismatch is allowed only where the oracle's choice scores nearly tie
        full = O.topk_by_choice(c[t], K)
        for k in range(K):
            a, b = int(idx_g[t, k]), int(idx_o[t, k])
            if a == b:
                continue
            if a < 0 or b < 0:  # top-p cut point moved: the running sums must straddle topp closely
                raw = s[t][full].astype(np.float64)
                cum = np.cumsum(raw / raw.sum())
                m = min(int(nsel_g[t]), int(n_o[t]))
                assert abs(cum[m - 1] - topp) < 1e-5, (t, cum, topp)
                break
            assert abs(float(c[t, a]) - float(c[t, b])) < NEAR_TIE, (t, k, a, b, c[t, a], c[t, b])
        near += 1
    return near, werr


def assert_close(got, ref, rtol, atol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    stats = dict(max_abs=float(err.max(initial=0)), max_rel=float((err / np.maximum(np.abs(ref), 1e-30)).max(initial=0)),
                 norm_rel=float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)), n_bad=int(bad.sum()))
    assert not bad.any(), f"{what}: {stats}; first bad at {np.argwhere(bad)[:5].tolist()}"
    return stats


def ffn_reference(cfg, x, idx, w, n_sel, resid):
    """Oracle FFN + reduce evaluated with the routes the GPU produced (no cascade of near-ties)."""
    experts = oracle_experts(cfg, idx)
    return O.expert_group(x, experts, idx, w, n_sel, resid)


class Ctx:
    def __init__(self, device=0):
        self.ctx = B.coli_init(device)

    @staticmethod
    def with_env(**env) -> "Ctx":
        """A context created while the given COLI_* variables are set (coli_init reads them)."""
        import os
        old = {k: os.environ.get(k) for k in env}
        os.environ.update({k: str(v) for k, v in env.items()})
        try:
            return Ctx()
        finally:
            for k, v in old.items():
                if v is None:
                    del os.environ[k]
                else:
                    os.environ[k] = v

    def close(self):
        if self.ctx is not None:
            B.coli_destroy(self.ctx)
            self.ctx = None
