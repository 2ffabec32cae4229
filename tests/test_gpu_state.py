"""GPU parity of the state-only pass (``la_state_pass``) and the ordered state sum
(``la_state_sum``) against the fp64 oracle.

``la_state_pass`` must end where the token recurrence ends after the same tokens:
``S_in + SiLU(K)^T SiLU(V)`` per (sequence, head) (oracle.state_pass, which a CPU pin
holds to the C token loop).  It is checked on shapes spanning several chunks and
segments with ragged tails, with and without an initial state, on already-activated
inputs, and on the 64-head 8K-token workload; ``la_state_sum`` must equal the fp32
left-to-right sum bit for bit.
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


def _kv(torch, B, N, H, seed):
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    _, k, v, _ = make_prefill_inputs(B, N, H, 128, torch.bfloat16, 0.5, seed, "cuda")
    return k, v


@pytest.mark.parametrize("with_state", [False, True])
@pytest.mark.parametrize("B,N,H", [(1, 1, 1), (1, 127, 2), (2, 300, 4), (1, 1000, 3),
                                   (3, 129, 8), (1, 2500, 64)])
def test_state_pass_matches_oracle(env, B, N, H, with_state):
    torch, la, orc = env
    from oracle.state_pass import state_pass
    k, v = _kv(torch, B, N, H, 5 + N + H)
    S_in = None
    if with_state:
        gen = torch.Generator(device="cuda").manual_seed(N + 1)
        S_in = torch.randn((B, H, 128, 128), generator=gen, device="cuda") * 0.5
    S = la.la_state_pass(k, v, kv_state_in=S_in)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    ref = state_pass(k.cpu(), v.cpu(), None if S_in is None else host64(S_in))
    ok, msg = state_ok(orc, host64(S), ref, host64(k), host64(v),
                       None if S_in is None else host64(S_in), "bf16")
    assert ok, msg
    # run to run: the same bits (segment states are added in a fixed order)
    S2 = la.la_state_pass(k, v, kv_state_in=S_in)
    torch.cuda.synchronize()
    assert torch.equal(S, S2)


def test_state_pass_in_place_and_empty(env):
    torch, la, orc = env
    from oracle.state_pass import state_pass
    k, v = _kv(torch, 2, 700, 4, 41)
    gen = torch.Generator(device="cuda").manual_seed(7)
    S = torch.randn((2, 4, 128, 128), generator=gen, device="cuda")
    S0 = host64(S)
    la.la_state_pass(k, v, kv_state_out=S, kv_state_in=S)  # continues in place
    torch.cuda.synchronize()
    ok, msg = state_ok(orc, host64(S), state_pass(k.cpu(), v.cpu(), S0), host64(k), host64(v),
                       S0, "bf16")
    assert ok, msg
    Z = la.la_state_pass(k[:, :0], v[:, :0])
    E = la.la_state_pass(k[:, :0], v[:, :0], kv_state_in=S)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Z) == 0 and torch.equal(E, S)


def test_state_pass_activated_inputs(env):
    """LA_FLAG_ACTIVATED: k and v arrive already SiLU-activated (as the input projection
    writes them); the pass then only sums K^T V."""
    torch, la, orc = env
    k, v = _kv(torch, 1, 900, 8, 77)
    ka = (k.float() * torch.sigmoid(k.float())).bfloat16()   # test-side activation
    va = (v.float() * torch.sigmoid(v.float())).bfloat16()
    S = la.la_state_pass(ka, va, activated=True)
    torch.cuda.synchronize()
    _, ref = orc.core(host64(ka), host64(ka), host64(va), want_y=False)
    assert rel_max_err(host64(S), ref) <= TOL["bf16"]["state"]


def test_state_pass_8k_workload(env):
    """B1 H64 N8192: the state the 8K prefill ends at, from k and v alone."""
    torch, la, orc = env
    from oracle.state_pass import state_pass
    from linear_attention_hybrid_fwd_b300.inputs import WORKLOADS, make_prefill_inputs
    w = WORKLOADS["prefill_8k"]
    q, k, v, g = make_prefill_inputs(w.B, w.N, w.H, w.d, torch.bfloat16, w.scale, w.seed,
                                     "cuda")
    S = la.la_state_pass(k, v)
    _, S_pre = la.la_prefill(q, k, v, g)
    torch.cuda.synchronize()
    ref = state_pass(k.cpu(), v.cpu())
    ok, msg = state_ok(orc, host64(S), ref, host64(k), host64(v), None, "bf16")
    assert ok, msg
    # the prefill's own final state: another summation order of the same sum
    assert rel_max_err(host64(S), host64(S_pre)) <= TOL["bf16"]["state"]


def test_state_sum_is_the_ordered_fp32_sum(env):
    torch, la, _ = env
    gen = torch.Generator(device="cuda").manual_seed(3)
    parts = torch.randn((5, 3, 2, 128, 128), generator=gen, device="cuda")
    base = torch.randn((3, 2, 128, 128), generator=gen, device="cuda")
    out = la.la_state_sum(parts, base=base)
    none = la.la_state_sum(parts[:0], base=base)
    nobase = la.la_state_sum(parts)
    torch.cuda.synchronize()
    acc = base.cpu().numpy().astype(np.float32)
    for p in parts.cpu().numpy():
        acc = acc + p                        # fp32 adds, left to right
    assert np.array_equal(out.cpu().numpy(), acc)
    assert torch.equal(none, base)
    acc0 = np.zeros_like(acc)
    for p in parts.cpu().numpy():
        acc0 = acc0 + p
    assert np.array_equal(nobase.cpu().numpy(), acc0)
