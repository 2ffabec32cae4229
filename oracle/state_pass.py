"""fp64 state pass over long sequences (test infrastructure, CPU only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
use this module; the CUDA library neither imports it nor shares code with it.

What it computes ("Hybrid Modeling", MiniMax-01 deep dive, Hugging Face blog: step 2
``K, V = SiLU(X)`` and step 3's ``K^T V``, the d x d state of the O(d^2 n) route): the
state after a run of tokens,

    S = S0 + sum_t SiLU(k_t)^T SiLU(v_t)        per (sequence b, head h),

which is exactly where the token recurrence S_t = S_{t-1} + k^_t^T v^_t ends.  It is
written with plain PyTorch CPU operations in fp64 (the textbook SiLU, then one batched
matrix product per call) so that the million-token workloads can be checked in
seconds; the C oracle's token loop computes the same sum one token at a time, and a
pin test holds the two to 1e-12.
"""
from __future__ import annotations

import numpy as np


def silu64(x):
    """SiLU(x) = x / (1 + e^-x), fp64 torch CPU tensor in, fp64 out."""
    import torch
    x = torch.as_tensor(x, dtype=torch.float64)
    return x / (1.0 + torch.exp(-x))


def state_pass(k, v, S0=None):
    """``k, v``: raw (pre-activation) ``[B, n, H, d]``; ``S0``: ``[B, H, d, d]`` or None.
    Returns the fp64 numpy state ``S0 + SiLU(K)^T SiLU(V)`` of shape ``[B, H, d, d]``."""
    import torch
    kh = silu64(k)
    vh = silu64(v)
    # [B, n, H, d] -> [B, H, d, n] @ [B, H, n, d]
    S = torch.einsum("bnhi,bnhj->bhij", kh, vh)
    if S0 is not None:
        S = S + torch.as_tensor(np.asarray(S0), dtype=torch.float64)
    return S.numpy()
