"""Run a synthetic MoE decode layer through the C ABI for a number of tokens and report timing.

    python -m int4_grouped_expert_router_gb300.run_layer --workload decode [--experts E] [--steps N]
    python -m int4_grouped_expert_router_gb300.run_layer --dense D [--tokens S] [--steps N]

Uploads the named workload's experts (optionally only the first E of them), then runs
coli_router_select + coli_expert_group per token, checks the device error word and prints the
mean event-timed microseconds per layer. With --dense D it instead runs coli_w4_linear through a
D x D per-row-scaled int4 tensor for S tokens per step. Used as the profiling target for single
kernels.
"""
from __future__ import annotations

import argparse
import dataclasses
import sys

import torch

from . import binding as B
from .build import build
from .workload import CONFIGS, DeviceLayer, router_host_inputs


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="decode", choices=sorted(CONFIGS))
    ap.add_argument("--experts", type=int, default=0, help="use only the first E experts")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--dense", type=int, default=0, help="time coli_w4_linear on a D x D tensor instead")
    ap.add_argument("--tokens", type=int, default=1, help="tokens per dense projection")
    args = ap.parse_args(argv)
    build()
    if args.dense:
        return run_dense(args.dense, args.tokens, args.warmup, args.steps)
    cfg = CONFIGS[args.workload]
    if args.experts:
        cfg = dataclasses.replace(cfg, E=args.experts, K=min(cfg.K, args.experts))
    ctx = B.coli_init(0)
    layer = DeviceLayer(ctx, cfg)
    stream = torch.cuda.current_stream()
    times = []
    for s in range(args.warmup + args.steps):
        x, _, _, resid = router_host_inputs(cfg, s)
        xt, rt = layer.act_tensor(x), layer.act_tensor(resid)
        out = layer.outputs()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer.step(xt, rt, out)
        b.record(stream)
        b.synchronize()
        if s >= args.warmup:
            times.append(a.elapsed_time(b) * 1000.0)
    rc = B.coli_check_error(ctx)
    layer.free()
    B.coli_destroy(ctx)
    if rc != 0:
        print(f"device error {rc}", file=sys.stderr)
        return 1
    print(f"{cfg.name} E={cfg.E}: {len(times)} steps, mean {sum(times) / len(times):.2f} us/layer")
    return 0


def run_dense(D, S, warmup, steps):
    from . import synth
    ctx = B.coli_init(0)
    p, sc = synth.expert_tensor_torch(synth.stream_seed(900, "dense"), D, D, 0, "cuda")
    h = B.coli_expert_upload(ctx, p.contiguous(), sc.contiguous(), D, D, 0)
    del p, sc
    stream = torch.cuda.current_stream()
    times = []
    for s in range(warmup + steps):
        x = torch.from_numpy(synth.normal(synth.stream_seed(901, s), S * D).reshape(S, D)).cuda()
        r = torch.from_numpy(synth.normal(synth.stream_seed(902, s), S * D).reshape(S, D)).cuda()
        y = torch.empty(S, D, device="cuda")
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        B.coli_w4_linear(ctx, h, x, r, y)
        b.record(stream)
        b.synchronize()
        if s >= warmup:
            times.append(a.elapsed_time(b) * 1000.0)
    rc = B.coli_check_error(ctx)
    B.coli_expert_free(ctx, h)
    B.coli_destroy(ctx)
    if rc != 0:
        print(f"device error {rc}", file=sys.stderr)
        return 1
    print(f"dense {D}x{D} S={S}: {len(times)} steps, mean {sum(times) / len(times):.2f} us")
    return 0


if __name__ == "__main__":
    sys.exit(main())
