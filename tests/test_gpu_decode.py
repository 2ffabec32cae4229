"""GPU parity of la_decode_step against the fp64 oracle recurrence.

The batched workload: B=256 sequences, 64 heads of 128, 64 steps, starting from the
state of a 1024-token bf16 prefill.  The oracle starts from that same fp32 state
(widened) and carries its own fp64 state through the 64 steps; every step's output
and the final state are compared.  The starting prefill itself is checked against
the oracle on 4 of the 256 sequences (all heads).
"""
import numpy as np
import pytest

from parity_util import TOL, host64, rel_max_err, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    la.load_library()
    return torch, la, oracle_mod


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_decode_small(env, dt):
    torch, la, orc = env
    from linear_attention_hybrid_fwd_b300.inputs import make_decode_inputs
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    B, H = 3, 5
    gen = torch.Generator(device="cuda").manual_seed(5)
    S = torch.randn((B, H, 128, 128), generator=gen, device="cuda") * 0.3
    S_ref = host64(S)
    y = torch.empty((B, H, 128), device="cuda")
    for step in range(6):
        q, k, v, g = make_decode_inputs(B, H, 128, dtype, 0.5, 77, step, "cuda")
        out = la.la_decode_step(S, q, k, v, g, y_debug=y)
        torch.cuda.synchronize()
        ref_out, ref_y, S_ref = orc.decode_step(S_ref, host64(q), host64(k), host64(v),
                                                host64(g))
        assert rel_max_err(host64(out), ref_out) <= TOL[dt]["out"]
        assert row_rel_err(host64(y), ref_y) <= TOL[dt]["y_row"]
        assert rel_max_err(host64(S), S_ref) <= TOL[dt]["state"]
    assert tuple(S.shape) == (B, H, 128, 128) and tuple(out.shape) == (B, H, 128)


@pytest.mark.parametrize("simt", [False, True])
def test_prefill_state_equals_decode_steps(env, simt):
    """GPU vs GPU: a prefill of N tokens and N decode steps give the same state and
    the same per-token outputs."""
    torch, la, _ = env
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    B, N, H = 2, 37, 4
    q, k, v, g = make_prefill_inputs(B, N, H, 128, torch.bfloat16, 0.5, 81, "cuda")
    out, S = la.la_prefill(q, k, v, g, simt=simt)
    Sd = torch.zeros_like(S)
    for t in range(N):
        o = la.la_decode_step(Sd, q[:, t].contiguous(), k[:, t].contiguous(),
                              v[:, t].contiguous(), g[:, t].contiguous())
        assert rel_max_err(host64(o), host64(out[:, t])) <= 1e-2
    torch.cuda.synchronize()
    # the tensor-core prefill forms k^T v from bf16-rounded operands; the decode kernel
    # and the CUDA-core prefill stay in fp32
    tol = 1e-5 if simt else TOL["bf16"]["state"]
    assert rel_max_err(host64(Sd), host64(S)) <= tol


def test_decode_b256_workload(env):
    torch, la, orc = env
    from linear_attention_hybrid_fwd_b300.inputs import (WORKLOADS, make_decode_inputs,
                                                         make_prefill_inputs)
    w = WORKLOADS["decode_b256"]
    q, k, v, g = make_prefill_inputs(w.B, w.N, w.H, w.d, torch.bfloat16, w.scale, w.seed,
                                     "cuda")
    _, S = la.la_prefill(q, k, v, g)
    torch.cuda.synchronize()
    # the starting prefill, checked on 4 seeded sequences (all heads)
    rows = np.random.default_rng(w.seed).choice(w.B, size=4, replace=False)
    for b in rows:
        sl = slice(int(b), int(b) + 1)
        ref_out, _, ref_S = orc.prefill(host64(q[sl]), host64(k[sl]), host64(v[sl]),
                                        host64(g[sl]))
        assert rel_max_err(host64(S[sl]), ref_S) <= TOL["bf16"]["state"]
    del q, k, v, g
    S_ref = host64(S)
    for step in range(w.decode_steps):
        q, k, v, g = make_decode_inputs(w.B, w.H, w.d, torch.bfloat16, w.scale, w.seed, step,
                                        "cuda")
        out = la.la_decode_step(S, q, k, v, g)
        torch.cuda.synchronize()
        ref_out, _, S_ref = orc.decode_step(S_ref, host64(q), host64(k), host64(v), host64(g))
        e = rel_max_err(host64(out), ref_out)
        assert e <= TOL["bf16"]["out"], f"step {step}: out rel err {e:.3e}"
    assert rel_max_err(host64(S), S_ref) <= TOL["bf16"]["state"]
    assert tuple(S.shape) == (w.B, w.H, w.d, w.d)
