"""Tensor-parallel MoE layer over R ranks, one GPU each (GLM-5.2 x10,
bandwidth model: TP8 splits every expert over 8 cards, so that each card
streams 1/8 of a layer's weight bytes).

Rank r holds, for every expert, the I-slice [r*I/R, (r+1)*I/R) of gate_up's
gate rows and of its up rows, and the same K-slice of down
(moeq_tp_shard_weights).  One layer step on a rank:
  1. moeq_moe_layer_shard: the full routing and live quantisation of x, the
     rank's h groups and their quantisation, and down over the rank's K
     slice, into an fp32 partial out [M, H];
  2. an all-gather of the partials, rank order kept, into [R, M, H];
  3. moeq_tp_reduce: out = bf16(partial_0 + partial_1 + ... in rank order),
     the same bits on every rank.
Step 2 is the one exchange; it goes through torch.distributed (NCCL between
GPUs), with plain device memory -- no multicast.  Each step can be replaced
(partial_fn, gather_fn, reduce_fn) so that the orchestration runs on CPU
ranks too.
"""
from __future__ import annotations

import torch

from . import moeq


class TPShard:
    """Rank `rank`'s shard of one layer's weights (E_total experts, the
    shared one included), cut on the device from the full tile-major
    weights."""

    def __init__(self, E_total: int, H: int, I: int, R: int, rank: int, w_gu, s_gu, w_d, s_d, stream=None):
        if I % (128 * R):
            raise ValueError(f"I = {I} does not split into {R} slices of whole 128-wide groups")
        self.E, self.H, self.I, self.R, self.rank, self.I_shard = E_total, H, I, R, rank, I // R
        dev = w_gu.device
        Is = self.I_shard
        self.w_gu = torch.empty((E_total, 2 * Is, H), dtype=torch.uint8, device=dev)
        self.s_gu = torch.empty((E_total, 2 * Is // 128, H // 128), dtype=torch.float32, device=dev)
        self.w_d = torch.empty((E_total, H, Is), dtype=torch.uint8, device=dev)
        self.s_d = torch.empty((E_total, H // 128, Is // 128), dtype=torch.float32, device=dev)
        moeq.moeq_tp_shard_weights(E_total, H, I, R, rank, w_gu, s_gu, w_d, s_d,
                                   self.w_gu, self.s_gu, self.w_d, self.s_d, stream=stream)


def gather_partials(partial: torch.Tensor, R: int, group=None) -> torch.Tensor:
    """All-gather of every rank's [M, H] partial into [R, M, H], in rank order."""
    import torch.distributed as dist
    parts = [torch.empty_like(partial) for _ in range(R)]
    dist.all_gather(parts, partial, group=group)
    return torch.stack(parts)


def tp_moe_layer(x, logits, E_routed: int, top_k: int, shard: TPShard, out, ws: moeq.Workspace, group=None,
                 partial_fn=None, gather_fn=None, reduce_fn=None):
    """One tensor-parallel layer step on this rank; `out` [M, H] bf16 gets
    the layer's output (identical on every rank).  Returns the gathered
    partials [R, M, H]."""
    M, H = x.shape
    partial = torch.empty((M, H), dtype=torch.float32, device=x.device)
    if partial_fn is None:
        moeq.moeq_moe_layer_shard(x, logits, H, shard.I_shard, E_routed, top_k, shard.w_gu, shard.s_gu,
                                  shard.w_d, shard.s_d, partial, ws)
    else:
        partial_fn(partial)
    parts = (gather_fn or gather_partials)(partial, shard.R, group)
    if reduce_fn is None:
        moeq.moeq_tp_reduce(parts, out)
    else:
        reduce_fn(parts, out)
    return parts
