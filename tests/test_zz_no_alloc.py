"""The decode step that allocates nothing (``la_decode_step_noalloc``).

Some callers cannot let a library call cudaMalloc: a serving engine that has reserved
all device memory for its own pool, or a latency-critical decode loop that cannot take
an allocation's device synchronisation.  For them the library runs the decode kernels
with their scratch in a fixed array of its own device data.  This test checks, through
the C ABI, that two calls in a row give what the allocating ``la_decode_step`` gives
on the same state and inputs, and that a batch beyond the array's size is refused
before anything is launched.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest

from parity_util import TOL, host64, rel_max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    la.load_library()
    return torch, la


@pytest.mark.parametrize("B,H", [(3, 5), (256, 64)])
def test_noalloc_matches_allocating_decode(env, B, H):
    torch, la = env
    from linear_attention_hybrid_fwd_b300.inputs import make_decode_inputs
    gen = torch.Generator(device="cuda").manual_seed(1234 + B)
    S_ref = torch.randn((B, H, 128, 128), generator=gen, device="cuda") * 0.3
    S_new = S_ref.clone()
    out_new = torch.empty((B, H, 128), device="cuda", dtype=torch.bfloat16)
    lib = la.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for step in range(2):  # two calls in a row: the scratch keeps the first call's data
        q, k, v, g = make_decode_inputs(B, H, 128, torch.bfloat16, 0.5, 91, step, "cuda")
        out_ref = la.la_decode_step(S_ref, q, k, v, g)
        rc = lib.la_decode_step_noalloc(
            ctypes.c_void_p(S_new.data_ptr()), ctypes.c_void_p(q.data_ptr()),
            ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(out_new.data_ptr()), B, H, 128,
            la.LA_BF16, 1e-6, stream)
        assert rc == la.LA_OK, la.la_status_string(rc)
        torch.cuda.synchronize()
        assert rel_max_err(host64(out_new), host64(out_ref)) <= TOL["bf16"]["out"]
        assert rel_max_err(host64(S_new), host64(S_ref)) <= TOL["bf16"]["state"]


def test_noalloc_refuses_batches_beyond_scratch(env):
    torch, la = env
    B, H = la.LA_NOALLOC_MAX_HEADS // 64 + 1, 64
    lib = la.load_library()
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(6)]  # never dereferenced
    rc = lib.la_decode_step_noalloc(p[0], p[1], p[2], p[3], p[4], p[5], B, H, 128,
                                    la.LA_BF16, 1e-6, None)
    assert rc == la.LA_ERR_SCRATCH_LIMIT
