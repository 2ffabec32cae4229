"""fp64 softmax attention with partial RoPE (test infrastructure, CPU only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
use this module; the CUDA library neither imports it nor shares code with it.

What it computes: the softmax layer that MiniMax-Text-01 places after every seven
Lightning Attention layers.  "Hybrid Modeling" (MiniMax-01 deep dive) notes that it
applies RoPE to only half of the head dimension.  The model card's "Model
Architecture" list gives 64 heads of size 128 and a RoPE base frequency of
10,000,000.  The deep dive's "10k base" is the first stage of its training schedule
("Long Context Training", which raises the base to 5M and then to 10M for the 1M-token
stage); the base is a parameter here, 1e7 by default.

Readings where the pages are silent:
* the rotated half is the first d/2 features of a head, rotated as d/4 pairs
  (i, i + d/4) ("rotate half"), with frequency theta_i = base^(-i / (d/4)) and angle
  t * theta_i at token position t = 0, 1, ...; the other d/2 features pass unchanged;
* scores are q_t . k_s / sqrt(d), causal (s <= t, the same inclusive causality as
  the linear layers), softmax over s, output sum_s p_ts v_s;
* every query head has its own key/value head (the pages name no grouping).
"""
from __future__ import annotations

import numpy as np


def rope(x, base=1.0e7, pos0=0):
    """``x``: [B, N, H, d] -> the same with its first d/2 features rotated (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    B, N, H, d = x.shape
    r = d // 4                                   # pairs in the rotated half
    theta = base ** (-np.arange(r, dtype=np.float64) / r)
    ang = (np.arange(N, dtype=np.float64) + pos0)[:, None] * theta[None, :]   # [N, r]
    c = np.cos(ang)[None, :, None, :]
    s = np.sin(ang)[None, :, None, :]
    a, b = x[..., :r], x[..., r:2 * r]
    out = x.copy()
    out[..., :r] = a * c - b * s
    out[..., r:2 * r] = a * s + b * c
    return out


def attention(q, k, v, base=1.0e7, causal=True):
    """Raw ``q, k, v`` [B, N, H, d] -> softmax(rope(q) rope(k)^T / sqrt(d)) v, fp64,
    computed one (b, h) score matrix at a time."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, N, H, d = q.shape
    qr, kr = rope(q, base), rope(k, base)
    out = np.empty((B, N, H, d))
    mask = np.triu(np.ones((N, N), dtype=bool), 1)          # s > t
    for b in range(B):
        for h in range(H):
            sc = qr[b, :, h] @ kr[b, :, h].T / np.sqrt(d)
            if causal:
                sc[mask] = -np.inf
            sc = sc - sc.max(axis=1, keepdims=True)
            p = np.exp(sc)
            p /= p.sum(axis=1, keepdims=True)
            out[b, :, h] = p @ v[b, :, h]
    return out
