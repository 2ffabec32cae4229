"""GPU parity of the packed ("varlen") prefill, la_prefill_varlen.

Sequences of different lengths, including empty ones and lengths that end mid-chunk,
are packed back to back.  Each sequence must equal its own la_prefill (bitwise on the
tensor-core kernel: the chunking of a sequence is the same) and the fp64 oracle run on
that sequence alone, for the output and the final state; an empty sequence's final
state is its initial state.
"""
import numpy as np
import pytest

from parity_util import TOL, host64, rel_max_err, state_ok

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


def _packed(torch, lens, H, dtype, seed):
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    cu = [0] + list(np.cumsum(lens))
    T = int(cu[-1])
    q, k, v, g = make_prefill_inputs(1, max(T, 1), H, 128, dtype, 0.5, seed, "cuda")
    return cu, [t[0, :T].contiguous() for t in (q, k, v, g)]


@pytest.mark.parametrize("H,lens,with_state", [
    (4, [300, 0, 1, 128, 129, 513], False),
    (4, [300, 0, 1, 128, 129, 513], True),
    (64, [1000, 77, 2048, 0, 3001], True),
    (8, [5], False),
])
def test_varlen_bf16(env, H, lens, with_state):
    torch, la, orc = env
    cu, (q, k, v, g) = _packed(torch, lens, H, torch.bfloat16, 7 + H + len(lens))
    S_in = None
    if with_state:
        gen = torch.Generator(device="cuda").manual_seed(31)
        S_in = torch.randn((len(lens), H, 128, 128), generator=gen, device="cuda") * 0.5
    out, S = la.la_prefill_varlen(q, k, v, g, cu, kv_state_in=S_in)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    assert la.la_prefill_path(1, H, int(cu[-1])) == 0
    for b, n in enumerate(lens):
        r0, r1 = int(cu[b]), int(cu[b + 1])
        if n == 0:
            want = torch.zeros_like(S[b]) if S_in is None else S_in[b]
            assert torch.equal(S[b], want)
            continue
        sl = [t[r0:r1].unsqueeze(0).contiguous() for t in (q, k, v, g)]
        o_b, S_b = la.la_prefill(*sl, kv_state_in=None if S_in is None else S_in[b:b + 1])
        torch.cuda.synchronize()
        assert torch.equal(out[r0:r1], o_b[0]), f"sequence {b}: differs from its own prefill"
        assert torch.equal(S[b], S_b[0]), f"sequence {b}: state differs from its own prefill"
        ref_out, _, ref_S = orc.prefill(*(host64(t) for t in sl),
                                        S0=None if S_in is None else host64(S_in[b:b + 1]))
        assert rel_max_err(host64(out[r0:r1]), ref_out[0]) <= TOL["bf16"]["out"]
        ok, msg = state_ok(orc, host64(S[b:b + 1]), ref_S, host64(sl[1]), host64(sl[2]),
                           None if S_in is None else host64(S_in[b:b + 1]), "bf16")
        assert ok, f"sequence {b}: {msg}"


def test_varlen_f32_cuda_core(env):
    torch, la, orc = env
    lens = [200, 0, 65]
    cu, (q, k, v, g) = _packed(torch, lens, 2, torch.float32, 12)
    out, S = la.la_prefill_varlen(q, k, v, g, cu)
    torch.cuda.synchronize()
    for b, n in enumerate(lens):
        r0, r1 = int(cu[b]), int(cu[b + 1])
        if n == 0:
            assert torch.count_nonzero(S[b]) == 0
            continue
        ref_out, _, ref_S = orc.prefill(*(host64(t[r0:r1]).reshape(1, n, 2, 128)
                                          for t in (q, k, v, g)))
        assert rel_max_err(host64(out[r0:r1]), ref_out[0]) <= TOL["f32"]["out"]
        ok, msg = state_ok(orc, host64(S[b:b + 1]), ref_S,
                           host64(k[r0:r1]).reshape(1, n, 2, 128),
                           host64(v[r0:r1]).reshape(1, n, 2, 128), None, "f32")
        assert ok, f"sequence {b}: {msg}"


def test_varlen_all_empty(env):
    torch, la, _ = env
    q = torch.empty((0, 4, 128), device="cuda", dtype=torch.bfloat16)
    S_in = torch.randn((3, 4, 128, 128), device="cuda")
    _, S = la.la_prefill_varlen(q, q, q, q, [0, 0, 0, 0], kv_state_in=S_in)
    torch.cuda.synchronize()
    assert torch.equal(S, S_in)


def test_varlen_bench_workload(env):
    """The packed batch bench.py times (64K tokens, H64, 15 sequences of seeded lengths
    in [1, 8192], one la_prefill_varlen launch): every sequence equals its own
    la_prefill bitwise; every final state matches the fp64 state pass; the output is
    checked against the oracle on the first 256 tokens of every sequence and on a
    256-token window at the end of two sequences (from the fp64 state before it)."""
    torch, la, orc = env
    from oracle.state_pass import state_pass
    from linear_attention_hybrid_fwd_b300.inputs import WORKLOADS, varlen_lengths
    w = WORKLOADS["prefill_varlen_64k"]
    lens = varlen_lengths(w.N, 1, 8192, w.seed)
    cu = [0] + [int(x) for x in np.cumsum(lens)]
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    q, k, v, g = (t[0] for t in make_prefill_inputs(1, w.N, w.H, w.d, torch.bfloat16,
                                                      w.scale, w.seed, "cuda"))
    out, S = la.la_prefill_varlen(q, k, v, g, cu)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    W = 256
    for b, n in enumerate(lens):
        r0, r1 = cu[b], cu[b + 1]
        sl = [t[r0:r1].unsqueeze(0).contiguous() for t in (q, k, v, g)]
        o_b, S_b = la.la_prefill(*sl)
        torch.cuda.synchronize()
        assert torch.equal(out[r0:r1], o_b[0]), f"sequence {b}: differs from its own prefill"
        assert torch.equal(S[b], S_b[0]), f"sequence {b}: state differs from its own prefill"
        S_ref = state_pass(sl[1].cpu(), sl[2].cpu())
        e_S = rel_max_err(host64(S[b:b + 1]), S_ref)
        assert e_S <= TOL["bf16"]["state"], f"sequence {b}: state rel err {e_S:.3e}"
        ref_out, _, _ = orc.prefill(*(host64(t[:, :W]) for t in sl))
        e = rel_max_err(host64(out[r0:r0 + W]), ref_out[0])
        assert e <= TOL["bf16"]["out"], f"sequence {b}: head window rel err {e:.3e}"
        if b in (0, len(lens) - 1):
            t0 = n - W
            S0 = state_pass(sl[1][:, :t0].cpu(), sl[2][:, :t0].cpu())
            ref_out, _, _ = orc.prefill(*(host64(t[:, t0:]) for t in sl), S0=S0)
            e = rel_max_err(host64(out[r0 + t0:r1]), ref_out[0])
            assert e <= TOL["bf16"]["out"], f"sequence {b}: tail window rel err {e:.3e}"
