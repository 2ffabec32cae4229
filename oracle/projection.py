"""fp64 input projection of the Lightning Attention layer (test infrastructure, CPU only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
use this module; the CUDA library neither imports it nor shares code with it.

What it computes.  "Hybrid Modeling" (MiniMax-01 deep dive, Hugging Face blog) lists
the mechanism as step 1 "Input X" and step 2 "Q, K, V = SiLU(X)"; the layer's input is
a token's hidden vector, 6144 wide in MiniMax-Text-01 (the model card's "Model
Architecture" list).  The step as printed omits the projections.  Reading: q, k, v and
the gate input g are four bias-free linear maps of x, and SiLU applies to q, k, v only
(g goes through sigmoid in step 4):

    q~ = x W_q^T,  k~ = x W_k^T,  v~ = x W_v^T,  g = x W_g^T
    activate:  q, k, v = SiLU(q~), SiLU(k~), SiLU(v~);  otherwise the raw q~, k~, v~

The four weight matrices are stacked into one [4*H*d, hidden] matrix W (rows
[0, Hd) for q, [Hd, 2Hd) for k, [2Hd, 3Hd) for v, [3Hd, 4Hd) for g; a fused
nn.Linear weight), and each output is reshaped to [T, H, d] (feature h*d + j is head
h, channel j).  The step is one library matrix product in fp64.
"""
from __future__ import annotations

import numpy as np


def silu(x):
    """SiLU(x) = x / (1 + e^-x) in fp64 (e^-x overflowing to inf gives -0)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def project(x, w, H, d, activate=True):
    """``x``: [T, hidden]; ``w``: [4*H*d, hidden].  Returns ``(q, k, v, g)``, each an
    fp64 array [T, H, d]; q, k, v are SiLU-activated when ``activate``."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, hidden = x.shape
    HD = H * d
    if w.shape != (4 * HD, hidden):
        raise ValueError(f"w must be [{4 * HD}, {hidden}], got {w.shape}")
    y = x @ w.T
    outs = [y[:, s * HD:(s + 1) * HD].reshape(T, H, d) for s in range(4)]
    if activate:
        outs = [silu(o) for o in outs[:3]] + [outs[3]]
    return tuple(outs)
