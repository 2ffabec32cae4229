"""GPU parity of the softmax layer (la_softmax_attention): partial RoPE + causal softmax
attention, against the fp64 oracle (oracle/softmax_attn.py) on the exact bf16 input
bits the GPU read.

Tolerance: max|out - ref| <= 1e-2 max|ref| per (sequence, head) slice, and the mean
error <= 2e-3 max|ref|.  The GPU rounds the rotated q and k to bf16 (2^-8 relative
each), the probabilities to bf16 for the P V product (2^-8), and the output once to
bf16 (2^-8); scores, the softmax statistics and the accumulation stay in fp32.  Each
output is a convex combination of v rows, so these relative roundings bound its error
by a few 2^-8 of max|v|-sized values; 1e-2 leaves about 2.5x headroom over 2^-8.
"""
import numpy as np
import pytest

from parity_util import host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    la.load_library()
    from oracle import softmax_attn
    return torch, la, softmax_attn


def _inputs(torch, B, N, H, seed):
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    q, k, v, _ = make_prefill_inputs(B, N, H, 128, torch.bfloat16, 1.0, seed, "cuda")
    return q, k, v


def _check(got, ref, heads=None):
    for b in range(ref.shape[0]):
        for h in (range(ref.shape[2]) if heads is None else heads):
            r = ref[b, :, h]
            g = got[b, :, h]
            den = np.abs(r).max()
            err = np.abs(g - r)
            assert err.max() <= 1e-2 * den, f"b{b} h{h}: max err {err.max() / den:.3e}"
            assert err.mean() <= 2e-3 * den, f"b{b} h{h}: mean err {err.mean() / den:.3e}"


@pytest.mark.parametrize("B,N,H", [(1, 1, 2), (1, 100, 2), (1, 128, 2), (2, 300, 2),
                                   (1, 1000, 4)])
def test_softmax_attention_small(env, B, N, H):
    torch, la, sa = env
    q, k, v = _inputs(torch, B, N, H, 50 + N)
    out = la.la_softmax_attention(q, k, v)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    _check(host64(out), sa.attention(host64(q), host64(k), host64(v)))


def test_softmax_attention_strong_rotation(env):
    """A small base rotates every pair fast, so a wrong pairing or sign shows."""
    torch, la, sa = env
    q, k, v = _inputs(torch, 1, 400, 2, 61)
    out = la.la_softmax_attention(q, k, v, rope_base=50.0)
    torch.cuda.synchronize()
    _check(host64(out), sa.attention(host64(q), host64(k), host64(v), base=50.0))


def test_softmax_attention_first_token_is_v0(env):
    torch, la, _ = env
    q, k, v = _inputs(torch, 2, 200, 3, 62)
    out = la.la_softmax_attention(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], v[:, 0])


def test_softmax_attention_8k_seeded_heads(env):
    """B1 H64 N8192 (the prefill workload's shape), the launch bench.py times; two seeded
    heads checked on every token against the oracle."""
    torch, la, sa = env
    from linear_attention_hybrid_fwd_b300.inputs import WORKLOADS
    w = WORKLOADS["attn_8k"]
    q, k, v = _inputs(torch, w.B, w.N, w.H, w.seed)
    out = la.la_softmax_attention(q, k, v)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    rng = np.random.default_rng(w.seed)
    for h in sorted(set(int(x) for x in rng.integers(0, w.H, 2))):
        sl = [host64(t[:, :, h:h + 1]) for t in (q, k, v)]
        _check(host64(out[:, :, h:h + 1]), sa.attention(*sl))
