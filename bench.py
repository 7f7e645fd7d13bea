#!/usr/bin/env python3
"""Benchmark of one decode-time MoE layer (device router + grouped int4 expert FFN + reduce).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload decode]

A step is one pass of the whole hot path for one token of the full-shape decode layer
(D=6144, I=2048, E=256 resident experts, K=8, S=1, per-row int4): coli_router_select followed by
coli_expert_group. Inputs are resident in HBM before the timed region. Each step is bracketed by
CUDA events on the library's stream; a 256 MiB buffer is written between steps (outside the
events) so every step starts with a cold L2. Rank 0 prints one JSON line.

--impl reference times the CPU oracle (the plain float64 restatement in oracle/) on the host's
cores for a bounded sample of the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per MoE decode layer (S=1, E=256,K=8) and expert-weight HBM GB/s vs peak"
UNIT = "us/layer"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill, shared-expert, dense-projection and compressed-tier figures")
    ap.add_argument("--parallel", default="ep", choices=["ep", "replicas"],
                    help="N > 1: split each layer's experts over the ranks (expert e on rank e mod N), or run N replicas")
    ap.add_argument("--cpu-steps", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-offset", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--check", default="", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-procs", type=int, default=0,
                    help="oracle processes of the CPU baseline (default: one per core this process may run on, at most 32)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def linear_leg(ctx, stream, flush, D, steps=20, warmup=3):
    """The dense int4 projection (coli_w4_linear) of one decode token through a D x D per-row-scaled
    tensor: event-timed launches with a cold L2, HBM bytes per launch and the fraction of the peak."""
    import numpy as np
    import torch

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300 import synth

    p, sc = synth.expert_tensor_torch(synth.stream_seed(900, "dense"), D, D, 0, "cuda")
    h = B.coli_expert_upload(ctx, p.contiguous(), sc.contiguous(), D, D, 0)
    del p, sc
    n = warmup + steps
    xs = [torch.from_numpy(synth.normal(synth.stream_seed(901, s), D).reshape(1, D)).cuda() for s in range(n)]
    rs = [torch.from_numpy(synth.normal(synth.stream_seed(902, s), D).reshape(1, D)).cuda() for s in range(n)]
    ys = [torch.empty(1, D, device="cuda") for _ in range(n)]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for s in range(n):
            flush.zero_()
            ev[s][0].record(stream)
            B.coli_w4_linear(ctx, h, xs[s], rs[s], ys[s])
            ev[s][1].record(stream)
    torch.cuda.synchronize()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    B.coli_expert_free(ctx, h)
    us = statistics.mean(ev[s][0].elapsed_time(ev[s][1]) for s in range(warmup, n)) * 1000.0
    nbytes = D * (D // 2) + 4 * D + 3 * 4 * D  # packed weights, row scales, x, resid, y
    hpeak, hkind = peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"dense int4 projection O={D} I={D} gs=0, S=1, f32, residual", "us": us, "steps": steps,
            "launch": "one C-ABI call per step", "l2": "flushed between steps", "bytes": nbytes, "hbm_gbs": gbs,
            "hbm_frac": gbs / hpeak, "peak_kind": f"{hkind} hbm_gbs"}


def ans_leg(ctx, stream, flush, nbytes, steps=10, warmup=3):
    """The compressed tier's decoder: one expert's gate + up packed bytes (quantised-weight-like nibbles)
    decoded from device-resident 4 KiB blocks, event-timed with a cold L2; raw bytes out per second."""
    import numpy as np
    import torch

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300 import synth

    data = synth.gaussian_nibble_bytes(synth.stream_seed(903, "tier"), nbytes, 2.5)
    h = B.coli_ans_upload(ctx, data.tobytes())
    raw, stored = B.coli_ans_info(ctx, h)
    out = torch.empty(raw, dtype=torch.uint8, device="cuda")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(warmup + steps)]
    with torch.cuda.stream(stream):
        for s in range(warmup + steps):
            flush.zero_()
            ev[s][0].record(stream)
            B.coli_ans_decode(ctx, h, out)
            ev[s][1].record(stream)
    torch.cuda.synchronize()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    ok = bool(np.array_equal(out.cpu().numpy(), data))
    B.coli_ans_free(ctx, h)
    us = statistics.mean(ev[s][0].elapsed_time(ev[s][1]) for s in range(warmup, warmup + steps)) * 1000.0
    return {"workload": f"{raw} bytes of packed int4 (nibbles ~ rounded N(7.5, 2.5^2)), 4 KiB rANS blocks",
            "us": us, "stored_over_raw": stored / raw, "raw_gbs": raw / (us * 1e-6) / 1e9,
            "stored_gbs": stored / (us * 1e-6) / 1e9, "exact": ok, "l2": "flushed between steps"}


def ans_gemv_leg(ctx, stream, flush, rows=2048, cols=6144, steps=10, warmup=3):
    """The compressed tier's fused block decode + GEMV on a gate-shaped tensor [2048 x 6144] (per-row scales,
    quantised-weight-like nibbles), beside decoding the same stream to a raw buffer and the raw int4 GEMV
    of the same tensor (uploaded uncompressed): event-timed, cold L2."""
    import numpy as np
    import torch

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300 import synth

    packed = synth.gaussian_nibble_bytes(synth.stream_seed(904, "tier-gemv"), rows * cols // 2, 2.5)
    scales = synth.uniform(synth.stream_seed(904, "tier-gemv-s"), rows, 0.005, 0.02).astype(np.float32)
    h = B.coli_ans_upload(ctx, packed.tobytes())
    raw, stored = B.coli_ans_info(ctx, h)
    W = B.coli_expert_upload(ctx, torch.from_numpy(packed), torch.from_numpy(scales), rows, cols, 0)
    st = torch.from_numpy(scales).cuda()
    x = torch.from_numpy(synth.normal(synth.stream_seed(904, "tier-gemv-x"), cols).astype(np.float32)).cuda()
    y_f, y_r = torch.empty(rows, device="cuda"), torch.empty(1, rows, device="cuda")
    out = torch.empty(raw, dtype=torch.uint8, device="cuda")
    calls = {"fused": lambda: B.coli_ans_w4_linear(ctx, h, st, rows, cols, 0, x, None, y_f),
             "decode_only": lambda: B.coli_ans_decode(ctx, h, out),
             "raw_gemv": lambda: B.coli_w4_linear(ctx, W, x.view(1, cols), None, y_r)}
    res = {}
    for name, call in calls.items():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(warmup + steps)]
        with torch.cuda.stream(stream):
            for s in range(warmup + steps):
                flush.zero_()
                ev[s][0].record(stream)
                call()
                ev[s][1].record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.mean(ev[s][0].elapsed_time(ev[s][1]) for s in range(warmup, warmup + steps)) * 1000.0
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    max_diff = float((y_f - y_r.view(-1)).abs().max().item())
    B.coli_ans_free(ctx, h)
    B.coli_expert_free(ctx, W)
    return {"workload": f"int4 [{rows} x {cols}], per-row scales, one token; stream of 4 KiB rANS blocks",
            "fused_us": res["fused"], "decode_only_us": res["decode_only"], "raw_gemv_us": res["raw_gemv"],
            "stored_over_raw": stored / raw, "fused_raw_gbs": raw / (res["fused"] * 1e-6) / 1e9,
            "max_abs_diff_fused_vs_raw_gemv": max_diff, "l2": "flushed between steps"}


def shared_expert_leg(ctx, stream, flush, layer, xs, rs, steps=20, warmup=3):
    """The decode layer with an always-chosen shared expert (weight 1, the routed experts' shape): the
    router appends it after the kept slots and one grouped call runs all K + 1 experts, as one CUDA
    graph per step."""
    import numpy as np
    import torch

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300 import synth
    from int4_grouped_expert_router_gb300.workload import tensor_seed

    cfg = layer.cfg
    e_sh = cfg.E  # outside the router's ids
    hs = []
    for which, (rows, cols) in (("gate", (cfg.I, cfg.D)), ("up", (cfg.I, cfg.D)), ("down", (cfg.D, cfg.I))):
        p, sc = synth.expert_tensor_torch(tensor_seed(cfg, e_sh, which), rows, cols, cfg.gs_of(e_sh), "cuda")
        hs.append(B.coli_expert_upload(ctx, p.contiguous(), sc.contiguous(), rows, cols, cfg.gs_of(e_sh)))
        del p, sc
    B.coli_expert_table_set(ctx, e_sh, *hs)
    xin, rin, yout = torch.empty_like(xs[0]), torch.empty_like(rs[0]), torch.empty_like(rs[0])
    r = dict(idx=torch.empty(cfg.S, cfg.K + 1, dtype=torch.int32, device="cuda"),
             w=torch.empty(cfg.S, cfg.K + 1, device="cuda"), n_sel=torch.empty(cfg.S, dtype=torch.int32, device="cuda"))

    def body():  # the router appends the shared slot; one grouped call runs the K + 1 experts
        B.coli_router_select_shared(ctx, xin, layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale,
                                    e_sh, r["idx"], r["w"], r["n_sel"])
        B.coli_expert_group(ctx, xin, r["idx"], r["w"], r["n_sel"], cfg.K + 1, rin, yout)

    n = min(len(xs), warmup + steps)
    with torch.cuda.stream(stream):
        xin.copy_(xs[0])
        rin.copy_(rs[0])
        body()  # eager once: the workspace is sized before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    routed_bytes = []
    with torch.cuda.stream(stream):
        for s in range(n):
            xin.copy_(xs[s])
            rin.copy_(rs[s])
            flush.zero_()
            ev[s][0].record(stream)
            g.replay()
            ev[s][1].record(stream)
            if s >= warmup:
                idx = r["idx"].cpu().numpy()
                routed_bytes.append(sum(cfg.expert_bytes(int(e)) for e in np.unique(idx[(idx >= 0) & (idx != e_sh)])))
    torch.cuda.synchronize()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    del g
    B.coli_expert_table_set(ctx, e_sh, 0, 0, 0)
    for h in hs:
        B.coli_expert_free(ctx, h)
    us = statistics.mean(ev[s][0].elapsed_time(ev[s][1]) for s in range(warmup, n)) * 1000.0
    nbytes = statistics.mean(routed_bytes) + cfg.expert_bytes(e_sh)
    hpeak, hkind = peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"decode layer + 1 shared expert (D={cfg.D} I={cfg.I}), K={cfg.K} routed of E={cfg.E}",
            "us_per_layer": us, "steps": n - warmup, "launch": "router with the shared slot + one grouped call of K+1 slots, one CUDA graph per step",
            "l2": "flushed between steps", "expert_bytes": nbytes, "hbm_gbs": gbs, "hbm_frac": gbs / hpeak,
            "peak_kind": f"{hkind} hbm_gbs"}


def prefill_leg(ctx, stream, flush, steps=10, warmup=3):
    """The prefill layer (S=512, g64 int4, bf16, Zipf routing) on the tensor-core path:
    graph-replayed steps with a cold L2, TFLOP/s and HBM bytes of the touched experts."""
    import numpy as np
    import torch

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300.workload import CONFIGS, DeviceLayer, router_host_inputs

    cfg = CONFIGS["prefill"]
    layer = DeviceLayer(ctx, cfg)
    n = warmup + steps
    xs, rs, outs = [], [], []
    for s in range(n):
        x, _, _, resid = router_host_inputs(cfg, 500000 + s)
        xs.append(layer.act_tensor(x))
        rs.append(layer.act_tensor(resid))
        outs.append(layer.outputs())
    for s in range(n):  # eager once (sizes the workspace), then one graph per step
        layer.step(xs[s], rs[s], outs[s])
    torch.cuda.synchronize()
    graphs = []
    for s in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            layer.step(xs[s], rs[s], outs[s])
        graphs.append(g)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for s in range(n):
        flush.zero_()
        ev[s][0].record(stream)
        graphs[s].replay()
        ev[s][1].record(stream)
    torch.cuda.synchronize()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(warmup, n)]
    del graphs
    B.coli_profile_enable(ctx, True)
    for k in (B.COLI_KERNEL_ROUTER, B.COLI_KERNEL_GATEUP, B.COLI_KERNEL_DOWN, B.COLI_KERNEL_COMBINE):
        B.coli_profile_read(ctx, k)
    for s in range(warmup, n):
        flush.zero_()
        layer.step(xs[s], rs[s], outs[s])
    kern = {}
    for name, k in (("router", B.COLI_KERNEL_ROUTER), ("gateup", B.COLI_KERNEL_GATEUP), ("down", B.COLI_KERNEL_DOWN),
                    ("combine", B.COLI_KERNEL_COMBINE)):
        t, c = B.coli_profile_read(ctx, k)
        if c:
            kern[name] = t * 1000.0 / c
    B.coli_profile_enable(ctx, False)
    routes, touched = [], []
    for s in range(warmup, n):
        idx = outs[s]["idx"].cpu().numpy()
        ids = idx[idx >= 0]
        routes.append(int(ids.size))
        touched.append(sum(cfg.expert_bytes(int(e)) for e in np.unique(ids)))
    layer.free()
    t_ms = statistics.mean(ms)
    flops = 6.0 * cfg.D * cfg.I * statistics.mean(routes)
    bpeak, bkind = bf16_peak()
    hpeak, hkind = peaks()
    tflops = flops / (t_ms * 1e-3) / 1e12
    gbs = statistics.mean(touched) / (t_ms * 1e-3) / 1e9
    mm_us = kern.get("gateup", 0.0) + kern.get("down", 0.0)
    return {
        "workload": f"prefill layer S={cfg.S} D={cfg.D} I={cfg.I} E={cfg.E} K={cfg.K}, int4 gs={cfg.gs}, bf16, Zipf routing",
        "ms_per_layer": t_ms, "steps": steps, "launch": "one CUDA graph per step", "l2": "flushed between steps",
        "routes": statistics.mean(routes), "gflop": flops / 1e9, "tflops": tflops,
        "tensor_frac": tflops / bpeak, "tensor_peak_tflops": bpeak, "tensor_peak_kind": f"{bkind} bf16_tflops",
        "expert_bytes": statistics.mean(touched), "hbm_gbs": gbs, "hbm_frac": gbs / hpeak,
        "gemm_tflops": flops / (mm_us * 1e-6) / 1e12 if mm_us else None, "kernels_us": kern,
    }


def decode_variant_leg(ctx, stream, flush, name, steps=20, warmup=3):
    """A decode-layer workload other than the headline one (the grouped-scale layer, or the S=4 bf16 Zipf
    layer): graph-replayed steps with a cold L2, per-kernel event means from a second pass, the distinct
    experts each step touched and the HBM fraction over their bytes."""
    import numpy as np
    import torch

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300.workload import CONFIGS, DeviceLayer, router_host_inputs

    cfg = CONFIGS[name]
    layer = DeviceLayer(ctx, cfg)
    B.coli_reserve(ctx, cfg.S, cfg.E, cfg.K, cfg.D, cfg.I)
    n = warmup + steps
    xs, rs, outs = [], [], []
    for s in range(n):
        x, _, _, resid = router_host_inputs(cfg, 700000 + s)
        xs.append(layer.act_tensor(x))
        rs.append(layer.act_tensor(resid))
        outs.append(layer.outputs())
    xin, rin, gout = torch.empty_like(xs[0]), torch.empty_like(rs[0]), layer.outputs()
    with torch.cuda.stream(stream):
        xin.copy_(xs[0])
        rin.copy_(rs[0])
        layer.step(xin, rin, gout)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer.step(xin, rin, gout)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for s in range(n):
            xin.copy_(xs[s])
            rin.copy_(rs[s])
            flush.zero_()
            ev[s][0].record(stream)
            g.replay()
            ev[s][1].record(stream)
            for k in ("idx", "w", "n_sel", "y"):
                outs[s][k].copy_(gout[k])
    torch.cuda.synchronize()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    del g
    us = [ev[s][0].elapsed_time(ev[s][1]) * 1000.0 for s in range(warmup, n)]
    B.coli_profile_enable(ctx, True)
    for k in (B.COLI_KERNEL_ROUTER, B.COLI_KERNEL_GATEUP, B.COLI_KERNEL_DOWN, B.COLI_KERNEL_COMBINE):
        B.coli_profile_read(ctx, k)
    with torch.cuda.stream(stream):
        for s in range(warmup, n):
            flush.zero_()
            layer.step(xs[s], rs[s], outs[s])
    kern = {}
    for kname, k in (("router", B.COLI_KERNEL_ROUTER), ("gateup_or_stream", B.COLI_KERNEL_GATEUP),
                     ("down", B.COLI_KERNEL_DOWN), ("combine_or_reduce", B.COLI_KERNEL_COMBINE)):
        t, c = B.coli_profile_read(ctx, k)
        if c:
            kern[kname] = t * 1000.0 / c
    B.coli_profile_enable(ctx, False)
    distinct, nbytes = [], []
    for s in range(warmup, n):
        idx = outs[s]["idx"].cpu().numpy()
        ids = np.unique(idx[idx >= 0])
        distinct.append(int(ids.size))
        nbytes.append(sum(cfg.expert_bytes(int(e)) for e in ids))
    layer.free()
    hpeak, hkind = peaks()
    mean_us = statistics.mean(us)
    gbs = statistics.mean(nbytes) / (mean_us * 1e-6) / 1e9
    return {"workload": workload_desc(cfg) + (", Zipf-skewed routing" if cfg.zipf else ""),
            "us_per_layer": mean_us, "p50_us": statistics.median(us), "steps": steps,
            "launch": "one CUDA graph (router + grouped call) per step", "l2": "flushed between steps",
            "kernels_us": kern, "distinct_experts": statistics.mean(distinct), "expert_bytes": statistics.mean(nbytes),
            "hbm_gbs": gbs, "hbm_frac": gbs / hpeak, "peak_kind": f"{hkind} hbm_gbs"}


def accuracy_sample(cfg, Wr, bias, xs_host, outs, rs_host, n_ffn=2):
    """Against the oracle, for the timed tokens: router near-ties (index disagreements allowed only where the
    oracle's choice scores are within 1e-6) over every timed token, and the largest |y - oracle| over the first
    n_ffn tokens (the oracle FFN evaluated with the GPU's routes), with the tolerance's absolute term."""
    import numpy as np

    import oracle.moe as O
    from int4_grouped_expert_router_gb300.workload import host_expert

    near, mismatch = 0, 0
    x_all = np.concatenate(xs_host, axis=0)
    idx_o, w_o, n_o, (_, _, c) = O.router_select(x_all, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
    for t, out in enumerate(outs):
        ig = np.asarray(out["idx"])[0]
        if np.array_equal(ig, idx_o[t]):
            continue
        # a disagreement is a near-tie when every differing pair of experts has choice scores within 1e-6
        pairs = [(int(a), int(b)) for a, b in zip(ig, idx_o[t]) if a != b and a >= 0 and b >= 0]
        if pairs and all(abs(float(c[t, a]) - float(c[t, b])) < 1e-6 for a, b in pairs):
            near += 1
        else:
            mismatch += 1
    max_err, atol = 0.0, None
    for t in range(min(n_ffn, len(outs))):
        ig, wg, ng, yg = (np.asarray(outs[t][k], dtype=np.float64) for k in ("idx", "w", "n_sel", "y"))
        ig = ig.astype(np.int32)
        wg = wg.astype(np.float32)
        ex = {}
        for e in sorted(set(int(v) for v in ig.reshape(-1) if v >= 0)):
            ex[e] = tuple(O.Tensor(p, s, r, cc, gs) for (p, s, r, cc, gs) in host_expert(cfg, e))
        ref = O.expert_group(xs_host[t], ex, ig, wg, ng.astype(np.int32), rs_host[t])
        max_err = max(max_err, float(np.abs(yg - ref).max()))
        rms = float(np.sqrt(np.mean(ref * ref)))
        atol = 1e-5 * max(1.0, rms)
    return {"tokens_routed": len(outs), "router_near_ties": near, "router_mismatches": mismatch,
            "ffn_tokens": min(n_ffn, len(outs)),
            "max_abs_err": max_err, "abs_term": atol,
            "tolerance": "rel 1e-4 + abs 1e-5 x max(1, rms(y)) per element"}


def ep_owned(e: int, rank: int, world: int) -> bool:
    """Expert parallelism: rank `rank` holds expert e when e mod world == rank."""
    return int(e) % int(world) == int(rank)


def ep_token_seed(step: int) -> int:
    """Under expert parallelism every rank works on the same token (each on its own experts)."""
    return token_seed(0, step)


def ep_job_us_per_layer(total_ms: float, steps: int) -> float:
    """Whole-job time per layer under expert parallelism: the ranks run the same `steps` layers together, so
    the job's time (the slowest rank's) is divided by the layers alone."""
    return total_ms * 1000.0 / steps


def token_seed(rank: int, step: int) -> int:
    """Seed of the token a rank processes at a step: every rank (replica) gets its own tokens."""
    return rank * 100000 + step


def max_over_ranks(value: float, dist, device: str) -> float:
    """The largest value over the ranks (the job takes as long as its slowest rank)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_layer(total_ms: float, steps: int, world: int) -> float:
    """Whole-job time per layer: every rank ran `steps` layers within `total_ms` (max over ranks)."""
    return total_ms * 1000.0 / (steps * world)


def workload_desc(cfg):
    return (f"MoE decode layer D={cfg.D} I={cfg.I} E={cfg.E} resident experts K={cfg.K} S={cfg.S}, "
            f"int4 gs={cfg.gs}, {cfg.x_dtype} activations, top-p={cfg.topp}")


# ------------------------------------------------------------------------------------------------
# CPU oracle leg (reference arm and cpu_baseline): runs in child processes, one per core, each pinned to one
# thread.
# ------------------------------------------------------------------------------------------------

def cpu_step_worker(workload: str, steps: int, warmup: int, check: str = "", offset: int = 0):
    """The oracle in steps of a bounded sample: step s routes token offset + s (the whole router) and runs
    ONE of its kept experts (slot s mod n_sel). The per-layer figure is the mean router time plus the mean
    kept count times the mean expert time."""
    import oracle.moe as O
    from int4_grouped_expert_router_gb300.workload import CONFIGS, host_expert, router_host_inputs

    cfg = CONFIGS[workload]
    t_router, t_expert, kept, t_step = [], [], [], []
    for s in range(warmup + steps):
        x, Wr, bias, resid = router_host_inputs(cfg, offset + s)
        t0 = time.perf_counter()
        idx, w, n, _ = O.router_select(x, Wr, bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale)
        t1 = time.perf_counter()
        k = s % int(n[0])
        gate, up, down = (O.Tensor(p, sc, r, c, gs) for (p, sc, r, c, gs) in host_expert(cfg, int(idx[0, k])))
        t2 = time.perf_counter()
        float(w[0, k]) * O.expert_ffn(x[0], gate, up, down)
        t3 = time.perf_counter()
        if s >= warmup:
            t_router.append(t1 - t0)
            t_expert.append(t3 - t2)
            kept.append(int(n[0]))
            t_step.append((t1 - t0) + (t3 - t2))
    mr, me, mk = statistics.mean(t_router), statistics.mean(t_expert), statistics.mean(kept)
    res = {"us_per_layer": (mr + mk * me) * 1e6, "steps": steps, "warmup": warmup,
           "ms_per_step": statistics.mean(t_step) * 1e3, "router_ms": mr * 1e3, "expert_ms": me * 1e3, "kept": mk}
    if check:  # the GPU arm's timed tokens, checked against the same oracle
        import numpy as np
        z = np.load(check)
        outs = [{"idx": z["idx"][t], "w": z["w"][t], "n_sel": z["n_sel"][t], "y": z["y"][t] if t < len(z["y"]) else None}
                for t in range(z["idx"].shape[0])]
        res["accuracy"] = accuracy_sample(cfg, z["Wr"], z["bias"], list(z["x"]), outs, list(z["resid"]),
                                          n_ffn=len(z["y"]))
    print(json.dumps(res))


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def combine_oracle_results(results):
    """Oracle processes run side by side on separate cores, each timing its own tokens: the box finishes
    layers at the sum of their rates, so its time per layer is 1 / sum(1 / t_i). Process 0's fields (and
    its accuracy check) are kept; `single_core_us` is the median single-process figure."""
    rate = sum(1.0 / r["us_per_layer"] for r in results)
    out = dict(results[0])
    out["us_per_layer"] = 1.0 / rate
    out["single_core_us"] = statistics.median(r["us_per_layer"] for r in results)
    out["procs"] = len(results)
    out["steps"] = sum(r["steps"] for r in results)
    out["router_ms"] = statistics.mean(r["router_ms"] for r in results)
    out["expert_ms"] = statistics.mean(r["expert_ms"] for r in results)
    out["kept"] = statistics.mean(r["kept"] for r in results)
    out["ms_per_step"] = statistics.mean(r["ms_per_step"] for r in results)
    return out


def run_oracle_steps(workload: str, steps: int, warmup: int, check: str = "", procs: int = 1):
    """cpu_step_worker in `procs` fresh single-threaded processes run at the same time (no GPU visible),
    each on its own tokens (process i starts at token 1000 i); only process 0 checks the GPU's tokens.
    Returns the combined JSON (combine_oracle_results)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    children = []
    for i in range(max(1, procs)):
        cmd = [sys.executable, os.path.abspath(__file__), "--cpu-steps", str(steps), "--warmup", str(warmup),
               "--workload", workload, "--cpu-offset", str(1000 * i)]
        if check and i == 0:
            cmd += ["--check", check]
        children.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env))
    results, errors = [], []
    for ch in children:
        try:
            out, err = ch.communicate(timeout=3600)
        except subprocess.TimeoutExpired:
            ch.kill()
            out, err = ch.communicate()
        if ch.returncode != 0:
            errors.append(err[-2000:])
        else:
            results.append(json.loads(out.strip().splitlines()[-1]))
    if errors or not results:
        raise RuntimeError(f"oracle timing failed: {(errors or ['no result'])[0]}")
    return combine_oracle_results(results)


def oracle_procs(args) -> int:
    return args.cpu_procs if args.cpu_procs > 0 else min(host_cores(), 32)


def oracle_sample(res, workload):
    procs = res.get("procs", 1)
    return (f"{procs} single-threaded oracle processes side by side, {res['steps']} steps in all, each one token of "
            f"the {workload} layer: the whole router and one of its kept experts in turn (router "
            f"{res['router_ms']:.1f} ms, expert {res['expert_ms']:.0f} ms, {res['kept']:.1f} kept); per process "
            f"router + kept x expert ({res.get('single_core_us', res['us_per_layer']) / 1000:.0f} ms per layer on one "
            "core); value = 1 / (sum of the processes' layer rates)")


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    from int4_grouped_expert_router_gb300.workload import CONFIGS
    cfg = CONFIGS[args.workload]
    try:
        res = run_oracle_steps(args.workload, args.steps, args.warmup, procs=oracle_procs(args))
    except RuntimeError:  # e.g. too little host memory for one process per core: one process
        res = run_oracle_steps(args.workload, args.steps, args.warmup, procs=1)
    v = res["us_per_layer"]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": res["warmup"], "ms_per_step": res["ms_per_step"], "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded SplitMix64; shapes of the pages' GLM-5.2 decode layer)",
        "config": {"workload": workload_desc(cfg)},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": res["procs"], "kind": "oracle",
                         "single_core_value": res["single_core_us"], "sample": oracle_sample(res, args.workload)},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, enabled=True):
        self.proc = None
        self.device_index = device_index
        if not enabled:
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={device_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def load_traffic(kernel: str, src_hash: str):
    """Per-launch DRAM bytes of ``kernel`` from the committed ncu summary, if taken on this source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if kv.get("kernel") == kernel and kv.get("source_sha") == src_hash:
                try:
                    return float(kv["dram_bytes_per_launch"])
                except (KeyError, ValueError):
                    return None
    return None


def source_hash():
    import hashlib
    h = hashlib.sha256()
    for name in ("experts.cu", "decode.cu", "dot.h", "coli_internal.h", "pipe.h"):
        with open(os.path.join(ROOT, "int4_grouped_expert_router_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def gpu_arm(args, rank, world, local):
    import numpy as np
    import torch

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300.build import build
    from int4_grouped_expert_router_gb300.workload import CONFIGS, DeviceLayer, router_host_inputs

    build()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cfg = CONFIGS[args.workload]
    stream = torch.cuda.Stream()  # a non-default stream: steps are captured into CUDA graphs
    torch.cuda.set_stream(stream)
    ctx = B.coli_init(local, stream)
    layer = DeviceLayer(ctx, cfg)
    n_tok = args.warmup + args.steps
    B.coli_reserve(ctx, cfg.S, cfg.E, cfg.K, cfg.D, cfg.I)

    # per-step inputs, resident on the device before timing (each rank its own tokens)
    xs, rs, xs_host, rs_host = [], [], [], []
    for s in range(n_tok):
        x, Wr_h, bias_h, resid = router_host_inputs(cfg, token_seed(rank, s))
        xs.append(layer.act_tensor(x))
        rs.append(layer.act_tensor(resid))
        xs_host.append(x)
        rs_host.append(resid)
    outs = [layer.outputs() for _ in range(n_tok)]
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    flush_sink = torch.empty(1, dtype=torch.float32, device="cuda")

    class _Flush:
        """Cold L2 for the next step: write 256 MiB (evicting everything), then read it back so
        the dirty lines are written back here, outside the timed events, and not by the step."""

        def zero_(self):
            flush_buf.zero_()
            torch.sum(flush_buf, dim=0, out=flush_sink[0])

    flush = _Flush()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_tok)]

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region: each step launches the two C-ABI calls (coli_router_select, coli_expert_group) as a
    # caller does, on inputs resident in HBM; before each step, outside its events, L2 is flushed ----
    for s in range(args.warmup):
        flush.zero_()
        layer.step(xs[s], rs[s], outs[s])
    barrier()
    clocks = ClockSampler(local, enabled=not args.no_clocks and rank == 0)
    time.sleep(0.3)
    t_wall = time.perf_counter()
    for s in range(args.warmup, n_tok):
        flush.zero_()
        ev[s][0].record(stream)
        layer.step(xs[s], rs[s], outs[s])
        ev[s][1].record(stream)
    barrier()
    wall = time.perf_counter() - t_wall
    clock_info = clocks.stop()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    step_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.warmup, n_tok)]

    # ---- the same steps replayed from one CUDA graph of the two calls over fixed device buffers, reported
    # beside (each step's inputs are copied in and L2 is flushed before its events) ----
    xin, rin, gout = torch.empty_like(xs[0]), torch.empty_like(rs[0]), layer.outputs()
    xin.copy_(xs[0])
    rin.copy_(rs[0])
    layer.step(xin, rin, gout)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layer.step(xin, rin, gout)
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_tok)]

    def graph_step(s):
        xin.copy_(xs[s])
        rin.copy_(rs[s])
        flush.zero_()
        gev[s][0].record(stream)
        graph.replay()
        gev[s][1].record(stream)

    for s in range(n_tok):
        graph_step(s)
    barrier()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    graph_ms = [gev[s][0].elapsed_time(gev[s][1]) for s in range(args.warmup, n_tok)]
    # back to back, reported beside the cold-L2 number: successive tokens' layers with no flush in between
    # (Wr and whatever else survives stays in L2); 8 graphs over 8 tokens' own buffers, replayed round robin
    # under one event pair
    n_b2b = 48
    b2b_graphs = []
    for i in range(8):
        gi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gi, stream=stream):
            layer.step(xs[args.warmup + i % args.steps], rs[args.warmup + i % args.steps], outs[args.warmup + i % args.steps])
        b2b_graphs.append(gi)
    torch.cuda.synchronize()
    b2b = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    b2b[0].record(stream)
    for i in range(n_b2b):
        b2b_graphs[i % 8].replay()
    b2b[1].record(stream)
    torch.cuda.synchronize()
    b2b_us = b2b[0].elapsed_time(b2b[1]) * 1000.0 / n_b2b
    del graph, b2b_graphs
    total_ms = max_over_ranks(sum(step_ms), dist, "cuda")
    us_per_layer = job_us_per_layer(total_ms, args.steps, world)

    # bytes each step had to read: the kept experts' packed weights + scales
    expert_bytes = []
    gateup_bytes = []
    for s in range(args.warmup, n_tok):
        idx = outs[s]["idx"].cpu().numpy()
        ids = [int(e) for e in idx.reshape(-1) if e >= 0]
        uniq = sorted(set(ids))
        expert_bytes.append(sum(cfg.expert_bytes(e) for e in uniq))
        gu = 0
        for e in uniq:
            gs = cfg.gs_of(e)
            from int4_grouped_expert_router_gb300 import synth
            gu += 2 * (cfg.I * ((cfg.D + 1) // 2) + 4 * synth.scale_count(cfg.I, cfg.D, gs))
        gateup_bytes.append(gu)
    mean_expert_bytes = float(np.mean(expert_bytes))
    hbm_peak, peak_kind = peaks()
    layer_gbs = mean_expert_bytes / (us_per_layer * 1e-6) / 1e9 * (1 if world == 1 else world)

    # ---- per-kernel durations: a second pass of the same steps with event pairs per launch ----
    B.coli_profile_enable(ctx, True)
    for k in (B.COLI_KERNEL_ROUTER, B.COLI_KERNEL_GATEUP, B.COLI_KERNEL_DOWN, B.COLI_KERNEL_COMBINE):
        B.coli_profile_read(ctx, k)
    for s in range(args.warmup, n_tok):
        flush.zero_()
        layer.step(xs[s], rs[s], outs[s])
    kern = {}
    for name, k in (("router", B.COLI_KERNEL_ROUTER), ("gateup", B.COLI_KERNEL_GATEUP), ("down", B.COLI_KERNEL_DOWN),
                    ("combine", B.COLI_KERNEL_COMBINE)):
        ms, n = B.coli_profile_read(ctx, k)
        if n:
            kern[name] = {"launches": n, "mean_us": ms * 1000.0 / n}
    B.coli_profile_enable(ctx, False)
    # S == 1 streams the whole expert FFN in one kernel (recorded as gate/up, no down launch; its reduce
    # is recorded as combine): its algorithmic bytes are every kept expert's gate, up and down bytes;
    # else the gate/up kernel's
    fused = "down" not in kern
    top_kernel = "stream_ffn_kernel" if fused else "gateup_kernel"
    top_bytes = float(np.mean(expert_bytes if fused else gateup_bytes))
    achieved = top_bytes / (kern["gateup"]["mean_us"] * 1e-6) / 1e9
    traffic = load_traffic(top_kernel, source_hash())

    # ---- end to end through the C ABI with host buffers: H2D inputs, D2H result per step ----
    # each step's x and resid sit side by side in one pinned host buffer and travel in one copy
    hxr = [torch.empty((2,) + tuple(xs[s].shape), dtype=xs[s].dtype, device="cpu").pin_memory() for s in range(n_tok)]
    hy = [torch.empty_like(outs[s]["y"], device="cpu").pin_memory() for s in range(n_tok)]
    for s in range(n_tok):
        hxr[s][0].copy_(xs[s])
        hxr[s][1].copy_(rs[s])
    dxr = [torch.empty((2,) + tuple(xs[s].shape), dtype=xs[s].dtype, device="cuda") for s in range(n_tok)]

    def e2e_step(s):
        dxr[s].copy_(hxr[s], non_blocking=True)
        layer.step(dxr[s][0], dxr[s][1], outs[s])
        hy[s].copy_(outs[s]["y"], non_blocking=True)

    for s in range(args.warmup):
        flush.zero_()
        e2e_step(s)
    barrier()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_tok)]
    for s in range(args.warmup, n_tok):
        flush.zero_()
        e2e_ev[s][0].record(stream)
        e2e_step(s)
        e2e_ev[s][1].record(stream)
    barrier()
    e2e_ms = max_over_ranks(sum(e2e_ev[s][0].elapsed_time(e2e_ev[s][1]) for s in range(args.warmup, n_tok)), dist, "cuda")
    e2e_us = job_us_per_layer(e2e_ms, args.steps, world)
    h2d = xs[0].numel() * xs[0].element_size() + rs[0].numel() * rs[0].element_size()
    d2h = outs[0]["y"].numel() * outs[0]["y"].element_size()

    # router + streaming FFN + its reduce, or router + gate/up + down (+ combine for S > 1)
    launches_per_step = 3 if fused else (3 if cfg.S == 1 else 4)
    result = None
    if rank == 0:
        cpu = None
        accuracy = None
        try:
            import tempfile
            timed = list(range(args.warmup, n_tok))
            n_ffn = min(2, len(timed))
            check = os.path.join(tempfile.mkdtemp(prefix="coli_bench_"), "timed.npz")
            np.savez(check, x=np.stack([xs_host[s] for s in timed]), resid=np.stack([rs_host[s] for s in timed]),
                     Wr=Wr_h, bias=bias_h, idx=np.stack([outs[s]["idx"].cpu().numpy() for s in timed]),
                     w=np.stack([outs[s]["w"].cpu().numpy() for s in timed]),
                     n_sel=np.stack([outs[s]["n_sel"].cpu().numpy() for s in timed]),
                     y=np.stack([outs[s]["y"].float().cpu().numpy() for s in timed[:n_ffn]]))
            # about 10 s of oracle on every core, and the check of the timed tokens against it
            res = run_oracle_steps(args.workload, 40, 1, check, procs=oracle_procs(args))
            accuracy = res.get("accuracy")
            cpu = {"value": res["us_per_layer"], "unit": UNIT, "cores": res["procs"], "kind": "oracle",
                   "single_core_value": res["single_core_us"], "sample": oracle_sample(res, args.workload)}
        except Exception as exc:  # the CPU leg must not hide the GPU number
            cpu = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {exc}"[:300]}
        p50 = statistics.median(step_ms) * 1000.0
        result = {
            "metric": METRIC, "value": us_per_layer, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us_per_layer / 1000.0 * world, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4xf32",
            "data": "synthetic (seeded SplitMix64; shapes of the pages' GLM-5.2 decode layer)",
            "config": {"workload": workload_desc(cfg), "l2": "flushed between steps (256 MiB write then read, outside the events)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "expert_bytes_per_layer": mean_expert_bytes,
                       "layer_hbm_gbs": layer_gbs, "layer_hbm_frac": layer_gbs / hbm_peak,
                       "launch": "coli_router_select + coli_expert_group launched per step (no graph), inputs resident in HBM",
                       "graph_us": statistics.mean(graph_ms) * 1000.0,
                       "graph": "the same two calls captured in one CUDA graph, replayed per step over fixed buffers into which each step's inputs are copied before its events",
                       "back_to_back_us": b2b_us, "back_to_back": "8 tokens' layer graphs replayed round robin, no L2 flush",
                       "p50_us": p50, "p10_us": float(np.percentile(step_ms, 10)) * 1000.0,
                       "p90_us": float(np.percentile(step_ms, 90)) * 1000.0,
                       "kernels_us": kern, "wall_s": wall},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic, "kernel": top_kernel,
                         "peak_kind": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": top_bytes},
            "cpu_baseline": cpu,
            "accuracy": accuracy,
            "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clock_info,
        }
    extra = {}
    if rank == 0 and not args.no_prefill:
        for name, leg in (("shared_expert", lambda: shared_expert_leg(ctx, stream, flush, layer, xs, rs)),
                          ("dense_projection", lambda: linear_leg(ctx, stream, flush, cfg.D)),
                          ("compressed_tier_decode", lambda: ans_leg(ctx, stream, flush, cfg.I * cfg.D)),
                          ("compressed_tier_gemv", lambda: ans_gemv_leg(ctx, stream, flush))):
            try:
                extra[name] = leg()
            except Exception as exc:  # these figures must not hide the decode number
                extra[name] = {"error": f"{exc}"[:300]}
    layer.free()
    # the other decode layers take the expert table over, so they run after the headline layer is freed
    if rank == 0 and not args.no_prefill:
        for name, leg in (("decode_grouped_scales", lambda: decode_variant_leg(ctx, stream, flush, "decode_g64")),
                          ("decode_s4_bf16_zipf", lambda: decode_variant_leg(ctx, stream, flush, "decode_s4_bf16"))):
            try:
                extra[name] = leg()
            except Exception as exc:  # these figures must not hide the decode number
                extra[name] = {"error": f"{exc}"[:300]}
    prefill = None
    if rank == 0 and not args.no_prefill:
        try:
            prefill = prefill_leg(ctx, stream, flush)
        except Exception as exc:  # the prefill figure must not hide the decode number
            prefill = {"error": f"{exc}"[:300]}
    if result is not None:
        result["prefill"] = prefill
        result.update(extra)
    B.coli_destroy(ctx)
    if dist is not None:
        dist.destroy_process_group()
    if result is not None:
        print(json.dumps(result))
    return 0


def ep_arm(args, rank, world, local):
    """N > 1, expert parallel: every rank routes the same tokens, runs its own experts' routes (issue + take),
    all-gathers the partial rows (NCCL) and adds them in rank order with the residual last. The job time per
    layer is the slowest rank's (strong scaling: the layer's work is fixed and split over the ranks)."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from int4_grouped_expert_router_gb300 import binding as B
    from int4_grouped_expert_router_gb300.build import build
    from int4_grouped_expert_router_gb300.ep import ExpertParallelLayer
    from int4_grouped_expert_router_gb300.workload import CONFIGS, DeviceLayer, router_host_inputs

    build()
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cfg = CONFIGS[args.workload]
    if cfg.x_dtype != "f32" or cfg.S != 1:
        raise SystemExit("the expert-parallel bench runs one f32 token per layer")
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    ctx = B.coli_init(local, stream)
    layer = DeviceLayer(ctx, cfg, owned=lambda e: ep_owned(e, rank, world))
    ep = ExpertParallelLayer(ctx, rank, world)
    n_tok = args.warmup + args.steps
    xs, rs = [], []
    for s in range(n_tok):
        x, _, _, resid = router_host_inputs(cfg, ep_token_seed(s))
        xs.append(layer.act_tensor(x))
        rs.append(layer.act_tensor(resid))
    y = torch.empty(1, cfg.D, device="cuda")
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    flush_sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def flush():
        flush_buf.zero_()
        torch.sum(flush_buf, dim=0, out=flush_sink[0])

    def step(s):
        return ep.step(xs[s], layer.Wr, layer.bias, cfg.K, cfg.topp, cfg.norm_topk, cfg.routed_scale, rs[s], y)

    for s in range(args.warmup):
        flush()
        step(s)
    dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_tok)]
    routes = []
    for s in range(args.warmup, n_tok):
        flush()
        ev[s][0].record(stream)
        idx, _, _ = step(s)
        ev[s][1].record(stream)
        routes.append(idx)
    dist.barrier()
    torch.cuda.synchronize()
    assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
    local_ms = sum(ev[s][0].elapsed_time(ev[s][1]) for s in range(args.warmup, n_tok))
    total_ms = max_over_ranks(local_ms, dist, "cuda")
    us = ep_job_us_per_layer(total_ms, args.steps)
    layer_bytes, my_bytes = [], []
    for idx in routes:
        ids = sorted(set(int(e) for e in idx.cpu().numpy().reshape(-1) if e >= 0))
        layer_bytes.append(sum(cfg.expert_bytes(e) for e in ids))
        my_bytes.append(sum(cfg.expert_bytes(e) for e in ids if ep_owned(e, rank, world)))
    hpeak, hkind = peaks()
    if rank == 0:
        gbs = float(np.mean(layer_bytes)) / (us * 1e-6) / 1e9
        print(json.dumps({
            "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1000.0, "higher_is_better": False, "scaling": "strong", "vs_baseline": None,
            "dtype": "int4xf32", "data": "synthetic (seeded SplitMix64; shapes of the pages' GLM-5.2 decode layer)",
            "config": {"workload": workload_desc(cfg), "parallelism": f"ep{world} (expert e on rank e mod {world})",
                       "l2": "flushed between steps (256 MiB write then read, outside the events)",
                       "launch": "router + routes shard + issue/take + NCCL all-gather + partials reduce per step",
                       "expert_bytes_per_layer": float(np.mean(layer_bytes)),
                       "rank0_expert_bytes_per_layer": float(np.mean(my_bytes)),
                       "layer_hbm_gbs": gbs, "layer_hbm_frac_of_one_gpu": gbs / hpeak},
        }))
    layer.free()
    B.coli_destroy(ctx)
    dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.cpu_steps:
        cpu_step_worker(args.workload, args.cpu_steps, args.warmup, args.check, args.cpu_offset)
        return 0
    rank, world, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if world > 1 and args.parallel == "ep":
        return ep_arm(args, rank, world, local)
    return gpu_arm(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
