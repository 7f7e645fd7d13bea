"""CPU oracle (test infrastructure only; see oracle/moe.py for its sources and readings)."""
from .moe import (  # noqa: F401
    F32, Tensor, dequant, expert_ffn, expert_group, pack_int4, route_weights, router_scores,
    router_select, scale_of, sigmoid64, silu64, topk_by_choice, unpack_int4,
)
