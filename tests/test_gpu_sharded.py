"""The sequence-sharded prefill's product path on one GPU: without a process group
(world size 1) it is exactly la_prefill, and its two-step form (a segment's state,
then the next segment continued from it through kv_state_in) matches the whole
sequence within the prefill's tolerances.  The exchange across ranks is tested with
gloo on CPU (test_sharded_cpu.py)."""
import pytest

from parity_util import TOL, host64, rel_max_err

pytestmark = pytest.mark.gpu


def test_sharded_prefill_single_rank_and_two_segments():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    from linear_attention_hybrid_fwd_b300.sharded import sharded_prefill
    q, k, v, g = make_prefill_inputs(1, 900, 4, 128, torch.bfloat16, 0.5, 91, "cuda")
    out1, S1 = sharded_prefill(q, k, v, g)
    ref_out, ref_S = la.la_prefill(q, k, v, g)
    torch.cuda.synchronize()
    assert torch.equal(out1, ref_out) and torch.equal(S1, ref_S)
    # two segments as two ranks would run them: 300 | 600 tokens
    seg = [t[:, :300].contiguous() for t in (q, k, v, g)]
    rest = [t[:, 300:].contiguous() for t in (q, k, v, g)]
    _, S_a = la.la_prefill(*seg)
    out_b, S_b = la.la_prefill(*rest, kv_state_in=S_a)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    assert rel_max_err(host64(out_b), host64(ref_out[:, 300:])) <= TOL["bf16"]["out"]
    assert rel_max_err(host64(S_b), host64(ref_S)) <= TOL["bf16"]["state"]
