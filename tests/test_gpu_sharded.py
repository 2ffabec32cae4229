"""The sequence-sharded prefill's product path on one GPU, against the fp64 oracle.

Without a process group (world size 1) ``sharded_prefill`` is exactly ``la_prefill``.
The steps W ranks run are replayed here on one GPU, segment by segment, with the
library's kernels: each segment's state from ``la_state_pass``, each prefix from
``la_state_sum`` in rank order, each segment's prefill from its prefix.  The
concatenated outputs and the final state must match the oracle on the whole sequence
within the prefill's tolerances.  The exchange itself (the all-gather across ranks) is
tested with gloo on CPU (test_sharded_cpu.py).
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


def test_sharded_prefill_single_rank_is_la_prefill(env):
    torch, la, _ = env
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    from linear_attention_hybrid_fwd_b300.sharded import sharded_prefill
    q, k, v, g = make_prefill_inputs(1, 900, 4, 128, torch.bfloat16, 0.5, 91, "cuda")
    out1, S1 = sharded_prefill(q, k, v, g)
    ref_out, ref_S = la.la_prefill(q, k, v, g)
    torch.cuda.synchronize()
    assert torch.equal(out1, ref_out) and torch.equal(S1, ref_S)


@pytest.mark.parametrize("segments", [[300, 600], [200, 350, 350], [129, 1, 770]])
def test_sharded_steps_match_oracle(env, segments):
    torch, la, orc = env
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    B, H, N = 2, 4, sum(segments)
    q, k, v, g = make_prefill_inputs(B, N, H, 128, torch.bfloat16, 0.5, 97, "cuda")
    bounds = np.cumsum([0] + segments)
    cut = lambda t, r: t[:, bounds[r]:bounds[r + 1]].contiguous()  # noqa: E731
    W = len(segments)
    # step 1 on every rank: its segment's own state (the last rank sends zeros)
    T = torch.stack([la.la_state_pass(cut(k, r), cut(v, r)) if r < W - 1 else
                     torch.zeros((B, H, 128, 128), device="cuda") for r in range(W)])
    outs, S_end = [], None
    for r in range(W):  # steps 3 and 4 on rank r
        prefix = la.la_state_sum(T[:r]) if r > 0 else None
        o, S_end = la.la_prefill(cut(q, r), cut(k, r), cut(v, r), cut(g, r),
                                 kv_state_in=prefix)
        outs.append(o)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    ref_out, _, ref_S = orc.prefill(host64(q), host64(k), host64(v), host64(g))
    assert rel_max_err(host64(torch.cat(outs, dim=1)), ref_out) <= TOL["bf16"]["out"]
    ok, msg = state_ok(orc, host64(S_end), ref_S, host64(k), host64(v), None, "bf16")
    assert ok, msg
