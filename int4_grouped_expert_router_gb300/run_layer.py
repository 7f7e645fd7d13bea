"""Run a synthetic MoE decode layer through the C ABI for a number of tokens and report timing.

    python -m int4_grouped_expert_router_gb300.run_layer --workload decode [--experts E] [--steps N]

Uploads the named workload's experts (optionally only the first E of them), then runs
coli_router_select + coli_expert_group per token, checks the device error word and prints the
mean event-timed microseconds per layer. Used as the profiling target for single kernels.
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
    args = ap.parse_args(argv)
    build()
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


if __name__ == "__main__":
    sys.exit(main())
