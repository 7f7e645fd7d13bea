"""Synthetic decode-layer workloads on the device: seeded experts uploaded through the C ABI.

The shapes and value distributions are those of the routed-expert layer the library targets
(D = 6144, I = 2048, E = 256, K = 8 at full size); weights are uniform nibbles with U(0.005, 0.02)
f32 scales, activations N(0, 1), router weights N(0, 0.02^2), biases U(-0.1, 0.1) or a
Zipf-skewed popularity bias. Every byte comes from int4_grouped_expert_router_gb300.synth, so the
same expert can be regenerated on the host for a reference computation.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import binding as B
from . import synth


@dataclasses.dataclass
class LayerConfig:
    name: str
    D: int
    I: int
    E: int
    K: int
    S: int = 1
    gs: object = 0            # int, or "mixed:<g>" (even experts gs=g, odd experts gs=0)
    x_dtype: str = "f32"      # "f32" or "bf16"
    topp: float = 0.0
    norm_topk: bool = True
    routed_scale: float = 2.5
    zipf: bool = False
    zipf_lambda: float = 0.25  # strength of the popularity bias (lambda ln p_rank)
    seed: int = synth.BASE_SEED

    def gs_of(self, e: int) -> int:
        if isinstance(self.gs, str) and self.gs.startswith("mixed:"):
            return int(self.gs.split(":")[1]) if e % 2 == 0 else 0
        return int(self.gs)

    def expert_bytes(self, e: int) -> int:
        """Packed weights + scales of expert e (the bytes one selection of it must read)."""
        gs = self.gs_of(e)
        n = 2 * self.I * ((self.D + 1) // 2) + self.D * ((self.I + 1) // 2)
        n += 4 * (2 * synth.scale_count(self.I, self.D, gs) + synth.scale_count(self.D, self.I, gs))
        return n


# Named workloads: the tiny correctness case and the full-shape decode variants.
CONFIGS = {
    "tiny": LayerConfig("tiny", D=256, I=128, E=16, K=4, routed_scale=2.5),
    "decode": LayerConfig("decode", D=6144, I=2048, E=256, K=8, routed_scale=2.5),
    "decode_g64": LayerConfig("decode_g64", D=6144, I=2048, E=256, K=8, gs="mixed:64", topp=0.9),
    "decode_g64_tail": LayerConfig("decode_g64_tail", D=6144, I=2000, E=256, K=8, gs=64, topp=0.9),
    "decode_s4_bf16": LayerConfig("decode_s4_bf16", D=6144, I=2048, E=256, K=8, S=4, x_dtype="bf16", zipf=True),
    # lambda 0.05: 4096 routes over ~150 experts, at most ~130 rows each (0.25 would put them on ~44)
    "prefill": LayerConfig("prefill", D=6144, I=2048, E=256, K=8, S=512, gs=64, x_dtype="bf16", zipf=True,
                           zipf_lambda=0.05),
}


def tensor_seed(cfg: LayerConfig, e: int, which: str) -> int:
    return synth.stream_seed(cfg.seed, "expert", e, which)


def host_expert(cfg: LayerConfig, e: int):
    """(gate, up, down) as numpy (packed, scales, rows, cols, gs) tuples, generated on the host."""
    gs = cfg.gs_of(e)
    out = []
    for which, (rows, cols) in (("gate", (cfg.I, cfg.D)), ("up", (cfg.I, cfg.D)), ("down", (cfg.D, cfg.I))):
        p, s = synth.expert_tensor(tensor_seed(cfg, e, which), rows, cols, gs)
        out.append((p, s, rows, cols, gs))
    return out


def router_host_inputs(cfg: LayerConfig, token0: int = 0):
    """x [S x D] f32 (bf16-representable when x_dtype is bf16), Wr [E x D], bias [E] for a batch."""
    _, Wr, bias = synth.router_inputs(cfg.seed, 1, cfg.D, cfg.E, zipf=cfg.zipf, zipf_lambda=cfg.zipf_lambda)
    x = synth.normal(synth.stream_seed(cfg.seed, "tokens", token0), cfg.S * cfg.D).reshape(cfg.S, cfg.D)
    if cfg.x_dtype == "bf16":
        x = synth.bf16_bits_to_f32(synth.to_bf16_bits(x))
    resid = synth.normal(synth.stream_seed(cfg.seed, "resid", token0), cfg.S * cfg.D).reshape(cfg.S, cfg.D)
    if cfg.x_dtype == "bf16":
        resid = synth.bf16_bits_to_f32(synth.to_bf16_bits(resid))
    return x, Wr, bias, resid


class DeviceLayer:
    """The E experts of one layer uploaded to the library (or only those `owned(e)` accepts: one rank's
    share under expert parallelism), plus device router weights."""

    def __init__(self, ctx, cfg: LayerConfig, device="cuda", generate_on_device=None, owned=None):
        self.ctx, self.cfg, self.device = ctx, cfg, device
        if generate_on_device is None:
            generate_on_device = cfg.D * cfg.I * cfg.E > 64 * 1024 * 1024
        self.handles = []
        for e in range(cfg.E):
            if owned is not None and not owned(e):
                self.handles.append(None)
                continue
            gs = cfg.gs_of(e)
            hs = []
            for which, (rows, cols) in (("gate", (cfg.I, cfg.D)), ("up", (cfg.I, cfg.D)), ("down", (cfg.D, cfg.I))):
                if generate_on_device:
                    p, s = synth.expert_tensor_torch(tensor_seed(cfg, e, which), rows, cols, gs, device)
                else:
                    pn, sn = synth.expert_tensor(tensor_seed(cfg, e, which), rows, cols, gs)
                    p, s = torch.from_numpy(pn), torch.from_numpy(sn)
                hs.append(B.coli_expert_upload(ctx, p.contiguous(), s.contiguous(), rows, cols, gs))
                del p, s
            B.coli_expert_table_set(ctx, e, *hs)
            self.handles.append(hs)
        _, Wr, bias = synth.router_inputs(cfg.seed, 1, cfg.D, cfg.E, zipf=cfg.zipf, zipf_lambda=cfg.zipf_lambda)
        self.Wr = torch.from_numpy(Wr).to(device)
        self.bias = torch.from_numpy(bias).to(device)

    def act_tensor(self, a: np.ndarray):
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(self.device)
        return t.to(torch.bfloat16) if self.cfg.x_dtype == "bf16" else t

    def outputs(self, S=None):
        S = S or self.cfg.S
        dt = torch.bfloat16 if self.cfg.x_dtype == "bf16" else torch.float32
        return dict(idx=torch.empty(S, self.cfg.K, dtype=torch.int32, device=self.device),
                    w=torch.empty(S, self.cfg.K, dtype=torch.float32, device=self.device),
                    n_sel=torch.empty(S, dtype=torch.int32, device=self.device),
                    y=torch.empty(S, self.cfg.D, dtype=dt, device=self.device))

    def step(self, x, resid, out):
        """One MoE layer: device router, then the grouped expert FFN with the weighted reduce."""
        c = self.cfg
        B.coli_router_select(self.ctx, x, self.Wr, self.bias, c.K, c.topp, c.norm_topk, c.routed_scale,
                             out["idx"], out["w"], out["n_sel"])
        B.coli_expert_group(self.ctx, x, out["idx"], out["w"], out["n_sel"], c.K, resid, out["y"])

    def free(self):
        for e, hs in enumerate(self.handles):
            if hs is not None:
                B.coli_expert_table_set(self.ctx, e, 0, 0, 0)
        for hs in self.handles:
            for h in hs or ():
                B.coli_expert_free(self.ctx, h)
        self.handles = []
