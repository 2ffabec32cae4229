"""Failure detection on the GPU without a fault: a cross-CTA arrival that never comes.

The tensor-core prefill's head pairs meet per chunk through counters in global memory
(the cross-head RMSNorm).  With LA_TEST_WITHHOLD_ARRIVAL=1 the library starts one
chunk's counter off its sentinel, as if one head half's arrival were lost.  Every wait
in the kernel is bounded: the launch must end with LA_ERR_TIMEOUT in the device status
word (and nothing else: no trap, no fault), and the next prefill on the same context
must be exactly the one a clean run gives.
"""
import os

import pytest

pytestmark = pytest.mark.gpu


def test_withheld_arrival_times_out_and_context_recovers():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    q, k, v, g = make_prefill_inputs(1, 1024, 4, 128, torch.bfloat16, 0.5, 71, "cuda")
    assert la.la_prefill_path(1, 4, 1024) == 0          # the tensor-core kernel
    ref_out, ref_S = la.la_prefill(q, k, v, g)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    os.environ["LA_TEST_WITHHOLD_ARRIVAL"] = "1"
    try:
        la.la_prefill(q, k, v, g)                        # the launch itself succeeds
        torch.cuda.synchronize()
    finally:
        del os.environ["LA_TEST_WITHHOLD_ARRIVAL"]
    assert la.la_get_device_status() == la.LA_ERR_TIMEOUT
    assert la.la_get_device_status() == 0                # reading clears it
    out, S = la.la_prefill(q, k, v, g)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    assert torch.equal(out, ref_out) and torch.equal(S, ref_S)
