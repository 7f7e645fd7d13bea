"""Expert parallelism across ranks (one process per GPU): the host orchestration around the device steps.

PR #434 "COLI_CUDA_RESID=1", section "What", reduces the expert groups' partial sums on the device in a fixed
order; the "GPU resident pipeline" commit of the c/backend_cuda.cu history spreads the expert groups over the
cards. Here expert e lives on rank e mod world. Every rank:

1. routes every token itself (coli_router_select is deterministic, so all ranks agree);
2. keeps the routes of its own experts (coli_routes_shard);
3. computes their weighted slot-order sum without the residual (coli_expert_group_issue + take, f32);
4. gathers every rank's partial rows in rank order (one all-gather, the only exchange);
5. adds them in rank order, the residual last (coli_partials_reduce): the same bits on every rank.

Each rank uploads only its own experts into its table; the expert ids stay global.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as B


def owner(e: int, world: int) -> int:
    """Rank holding expert e."""
    return int(e) % int(world)


def gather_partials(partial: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's partial rows stacked in rank order, [world x S x D] (the same stack on every rank)."""
    world = dist.get_world_size(group)
    parts = [torch.empty_like(partial) for _ in range(world)]
    dist.all_gather(parts, partial.contiguous(), group=group)
    return torch.stack(parts)


class ExpertParallelLayer:
    """One rank's side of an expert-parallel MoE block over a context whose table holds this rank's experts."""

    def __init__(self, ctx, rank: int, world: int, group=None):
        self.ctx, self.rank, self.world, self.group = ctx, rank, world, group

    def step(self, x, Wr, bias, K, topp, norm_topk, routed_scale, resid, y):
        if x.dtype != torch.float32:
            raise ValueError("expert-parallel partial sums are exchanged in f32: pass f32 activations")
        S = x.shape[0]
        dev = x.device
        idx = torch.empty(S, K, dtype=torch.int32, device=dev)
        w = torch.empty(S, K, dtype=torch.float32, device=dev)
        n = torch.empty(S, dtype=torch.int32, device=dev)
        B.coli_router_select(self.ctx, x, Wr, bias, K, topp, norm_topk, routed_scale, idx, w, n)
        idx_r, w_r, n_r = torch.empty_like(idx), torch.empty_like(w), torch.empty_like(n)
        B.coli_routes_shard(self.ctx, idx, w, n, self.rank, self.world, idx_r, w_r, n_r)
        partial = torch.empty(S, x.shape[1], dtype=torch.float32, device=dev)
        B.coli_expert_group_issue(self.ctx, x, idx_r, w_r, n_r, K)
        B.coli_expert_group_take(self.ctx, None, partial)
        parts = gather_partials(partial, self.group) if self.world > 1 else partial.unsqueeze(0)
        B.coli_partials_reduce(self.ctx, parts, resid, y)
        return idx, w, n
