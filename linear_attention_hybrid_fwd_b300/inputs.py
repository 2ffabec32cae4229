"""Seeded synthetic inputs and the workload shapes (no arithmetic of the method here).

Shapes follow the MiniMax-Text-01 architecture list (64 attention heads of size 128;
1M-token context).  There is no dataset and there are no trained weights: q, k, v, g
stand for the pre-activation projection outputs and are drawn i.i.d. normal.

Both the CUDA path (tests, bench) and the oracle side take their inputs from here:
the oracle gets host copies of exactly the bits the GPU saw.
"""
from __future__ import annotations

from dataclasses import dataclass

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "g": 3, "x": 4, "w": 5}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str        # "bf16" or "f32"
    scale: float      # inputs are N(0, 1) * scale before the cast
    seed: int
    decode_steps: int = 0
    hidden: int = 0   # input projection: width of the token's hidden vector


WORKLOADS = {
    # fp32 I/O, B1 H1 N512, N(0,1), seed 0; norm over the d features
    "tiny_f32": Workload("tiny_f32", 1, 1, 512, 128, "f32", 1.0, 0),
    # the 64 x 128-head prefill at 8K tokens
    "prefill_8k": Workload("prefill_8k", 1, 64, 8192, 128, "bf16", 0.5, 2),
    # long prefill, 128K tokens
    "prefill_128k": Workload("prefill_128k", 1, 64, 131072, 128, "bf16", 0.5, 3),
    # batched decode: 256 sequences x 64 steps from a 1024-token prefilled state
    "decode_b256": Workload("decode_b256", 256, 64, 1024, 128, "bf16", 0.5, 4, decode_steps=64),
    # 1M-token prefill
    "prefill_1m": Workload("prefill_1m", 1, 64, 1048576, 128, "bf16", 0.5, 5),
    # input projection of the 8K prefill: x [8192, 6144] -> q, k, v, g [8192, 64, 128]
    "proj_8k": Workload("proj_8k", 1, 64, 8192, 128, "bf16", 1.0, 7, hidden=6144),
    # the softmax layer at the 8K prefill's shape: q, k, v N(0,1), RoPE base 1e7
    "attn_8k": Workload("attn_8k", 1, 64, 8192, 128, "bf16", 1.0, 8),
    # packed batch: 64K tokens in sequences of seeded lengths (varlen_lengths)
    "prefill_varlen_64k": Workload("prefill_varlen_64k", 1, 64, 65536, 128, "bf16", 0.5, 6),
    # one long sequence with few heads (8 of 128): the segment-parallel prefill
    "prefill_h8_256k": Workload("prefill_h8_256k", 1, 8, 262144, 128, "bf16", 0.5, 9),
}


def varlen_lengths(total: int, lo: int, hi: int, seed: int):
    """Sequence lengths drawn uniformly from [lo, hi] (numpy default_rng(seed)) until
    they sum to ``total``; the last one is cut to fit.  Returns a list of ints."""
    import numpy as np
    rng = np.random.default_rng(seed)
    lens, left = [], total
    while left > 0:
        n = min(int(rng.integers(lo, hi + 1)), left)
        lens.append(n)
        left -= n
    return lens


def torch_dtype(name: str):
    import torch
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def make_tensor(shape, dtype, scale: float, seed: int, tensor_id: int, device,
                chunk_rows: int = 65536):
    """N(0,1)*scale, cast round-to-nearest-even to ``dtype``; generated in slabs of
    ``chunk_rows`` along axis 1 so fp32 temporaries stay small.  The generator is
    seeded with ``seed * 16 + tensor_id`` on ``device``."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 16 + tensor_id)
    out = torch.empty(shape, dtype=dtype, device=device)
    if len(shape) < 2 or shape[1] <= chunk_rows:
        out.copy_(torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * scale)
        return out
    for s in range(0, shape[1], chunk_rows):
        e = min(shape[1], s + chunk_rows)
        sub = (shape[0], e - s) + tuple(shape[2:])
        out[:, s:e].copy_(torch.randn(sub, generator=gen, device=device,
                                      dtype=torch.float32) * scale)
    return out


def make_prefill_inputs(B, N, H, d, dtype, scale, seed, device):
    """q, k, v, g of shape ``[B, N, H, d]``."""
    return tuple(make_tensor((B, N, H, d), dtype, scale, seed, TENSOR_IDS[n], device)
                 for n in ("q", "k", "v", "g"))


def make_projection_inputs(T, hidden, H, d, seed, device, wscale=None):
    """x ``[T, hidden]`` N(0,1) and the stacked weight ``[4*H*d, hidden]``
    N(0,1)*wscale (default 0.5/sqrt(hidden), so each projected feature is about
    N(0, 0.25), the spread of the prefill workloads' inputs), both bf16."""
    import torch
    if wscale is None:
        wscale = 0.5 / hidden ** 0.5
    x = make_tensor((1, T, hidden), torch.bfloat16, 1.0, seed, TENSOR_IDS["x"], device)[0]
    w = make_tensor((1, 4 * H * d, hidden), torch.bfloat16, wscale, seed, TENSOR_IDS["w"],
                    device)[0]
    return x, w


def make_decode_inputs(B, H, d, dtype, scale, seed, step, device):
    """q, k, v, g of shape ``[B, H, d]`` for decode step ``step``."""
    return tuple(make_tensor((B, H, d), dtype, scale, seed * 1000 + step, TENSOR_IDS[n],
                             device) for n in ("q", "k", "v", "g"))
