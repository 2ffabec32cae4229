"""Sequence-sharded prefill across ranks (one process per GPU).

What it computes: the same layer as ``la_prefill`` over one long sequence (per batch
row) whose tokens are split into contiguous segments, rank r holding segment r.  The
MiniMax-01 deep dive ("Post Training and Infra") names linear-attention sequence
parallelism among the infrastructure improvements without describing it; the plainest
scheme the method allows is used here.  Only the d x d state crosses a segment
boundary: with S_r the state of segment r alone (from zero),

    rank r's prefix state  P_r = S_0 + ... + S_{r-1}

and rank r's outputs are its segment's prefill continued from P_r (``kv_state_in``).
The RMSNorm spans a token's H*d features, all on one rank, so nothing else is
exchanged.

Steps per rank:
1. S_r: the segment's prefill from zero (``kv_state_out``);
2. P_r: one ``reduce`` per destination rank over the ranks before it (the collective
   does the fp32 additions; contributions from later ranks are zeros);
3. rank 0's outputs are those of step 1; every other rank runs its segment again
   from P_r.
Ranks after the first run their segment twice, so W ranks finish a sequence about
W/2 times faster than one; a state-only kernel would remove the first run.

``op`` is the per-rank prefill (default ``la_prefill``); tests pass a CPU stand-in to
check the exchange with the gloo backend.
"""
from __future__ import annotations


def sharded_prefill(q, k, v, g, group=None, op=None, eps: float = 1e-6):
    """``q, k, v, g``: this rank's segment ``[B, N_r, H, d]`` (segments in rank order).
    Returns ``(out, S_end)``: the segment's outputs and the state after its last token
    (on the last rank, the state of the whole sequence)."""
    import torch
    import torch.distributed as dist
    if op is None:
        from . import la_prefill as op
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    out, S_seg = op(q, k, v, g, eps=eps)
    if world == 1:
        return out, S_seg
    prefix = None
    for dst in range(1, world):
        buf = S_seg.clone() if rank < dst else torch.zeros_like(S_seg)
        dist.reduce(buf, dst=_global_rank(group, dst), op=dist.ReduceOp.SUM, group=group)
        if rank == dst:
            prefix = buf
    if rank == 0:
        return out, S_seg
    return op(q, k, v, g, kv_state_in=prefix, eps=eps)


def _global_rank(group, r):
    import torch.distributed as dist
    if group is None:
        return r
    return dist.get_global_rank(group, r)
