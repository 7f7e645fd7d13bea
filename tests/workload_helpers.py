"""Oracle-side helpers for tests that upload experts by hand."""
import numpy as np

import oracle.moe as O
from int4_grouped_expert_router_gb300 import synth


def oracle_for_layer_seed(cfg, x, idx, w, resid=None):
    experts = {}
    for e in sorted(set(int(v) for v in idx.reshape(-1) if v >= 0)):
        trip = []
        for which, (r, c) in (("gate", (cfg.I, cfg.D)), ("up", (cfg.I, cfg.D)), ("down", (cfg.D, cfg.I))):
            p, s = synth.expert_tensor(synth.stream_seed(cfg.seed, "expert", e, which), r, c, 0)
            trip.append(O.Tensor(p, s, r, c, 0))
        experts[e] = tuple(trip)
    return O.expert_group(x, experts, idx, w, None, resid)
