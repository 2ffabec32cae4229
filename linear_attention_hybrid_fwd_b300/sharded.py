"""Sequence-sharded prefill across ranks (one process per GPU).

What it computes: the same layer as ``la_prefill`` over one long sequence (per batch
row) whose tokens are split into contiguous segments, rank r holding segment r.  The
MiniMax-01 deep dive ("Post Training and Infra") names linear-attention sequence
parallelism among the infrastructure improvements without describing it; the plainest
scheme the method allows is used here.  Only the d x d state crosses a segment
boundary: with T_r = SiLU(K_r)^T SiLU(V_r) the state of segment r alone,

    rank r's prefix state  P_r = S_0 + T_0 + ... + T_{r-1}

and rank r's outputs are its segment's prefill continued from P_r (``kv_state_in``).
The RMSNorm spans a token's H*d features, all on one rank, so nothing else is
exchanged.

Steps per rank:
1. T_r with the state-only pass (``la_state_pass``: reads k and v only); the last rank's
   state is no rank's prefix, so it passes zero tokens and sends zeros;
2. one ``all_gather`` of the W states ([W, B, H, d, d] fp32: W * 4 MiB at B = 1, H = 64);
3. P_r = S_0 + T_0 + ... + T_{r-1}, added in rank order (``la_state_sum``), so every
   rank's prefix is the same fp32 sum whatever the collective's own reduction order;
4. the segment's prefill from P_r (``la_prefill``).
Per rank this moves the segment's k and v twice and q, g, out once: 7/5 of one
unsharded prefill of the segment, plus the all-gather.

``ops`` replaces the three per-rank operations (``prefill``, ``state_pass``,
``state_sum``); tests pass fp64 CPU stand-ins to check the exchange with the gloo
backend.
"""
from __future__ import annotations


def _library_ops():
    from . import la_prefill, la_state_pass, la_state_sum
    return {"prefill": la_prefill, "state_pass": la_state_pass, "state_sum": la_state_sum}


def sharded_prefill(q, k, v, g, group=None, ops=None, eps: float = 1e-6, S0=None):
    """``q, k, v, g``: this rank's segment ``[B, N_r, H, d]`` (segments in rank order);
    ``S0``: the state before the first segment (``[B, H, d, d]`` fp32, same on every
    rank) or None for zeros.  Returns ``(out, S_end)``: the segment's outputs and the
    state after its last token (on the last rank, the state of the whole sequence)."""
    import torch
    import torch.distributed as dist
    ops = dict(_library_ops(), **(ops or {}))
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    if world == 1:
        return ops["prefill"](q, k, v, g, kv_state_in=S0, eps=eps)
    # the last segment's state is no rank's prefix: that rank passes zero tokens
    T = ops["state_pass"](k, v) if rank < world - 1 else ops["state_pass"](k[:, :0], v[:, :0])
    gathered = [torch.empty_like(T) for _ in range(world)]
    dist.all_gather(gathered, T.contiguous(), group=group)
    if rank == 0:
        prefix = S0
    else:
        prefix = ops["state_sum"](torch.stack(gathered[:rank]), base=S0)
    return ops["prefill"](q, k, v, g, kv_state_in=prefix, eps=eps)
