"""The decode step that allocates nothing (``la_decode_step_noalloc``).

Some callers cannot let a library call cudaMalloc: a serving engine that has reserved
all device memory for its own pool, or a latency-critical decode loop that cannot take
an allocation's device synchronisation.  For them the library runs the decode kernels
with their scratch in a fixed array of its own device data.  This test checks, through
the C ABI, that two calls in a row give bit for bit what the allocating
``la_decode_step`` gives on the same state and inputs (both run the same kernel), that
those calls leave the device's free memory unchanged, and that a batch beyond the
array's size is refused before anything is launched.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest


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


def _noalloc(lib, la, S, q, k, v, g, out, B, H, stream):
    return lib.la_decode_step_noalloc(
        ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(out.data_ptr()), B, H, 128, la.LA_BF16,
        1e-6, stream)


@pytest.mark.parametrize("B,H", [(3, 5), (256, 64)])
def test_noalloc_matches_allocating_decode(env, B, H):
    torch, la = env
    from linear_attention_hybrid_fwd_b300.inputs import make_decode_inputs
    gen = torch.Generator(device="cuda").manual_seed(1234 + B)
    S0 = torch.randn((B, H, 128, 128), generator=gen, device="cuda") * 0.3
    steps = [make_decode_inputs(B, H, 128, torch.bfloat16, 0.5, 91, s, "cuda") for s in range(2)]
    S_new, S_warm = S0.clone(), S0.clone()
    outs = [torch.empty((B, H, 128), device="cuda", dtype=torch.bfloat16) for _ in range(3)]
    lib = la.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the first call on the device looks the scratch address up; after it, calls must
    # leave the device's free memory exactly where it was
    assert _noalloc(lib, la, S_warm, *steps[0], outs[2], B, H, stream) == la.LA_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for step in range(2):  # two calls in a row: the scratch keeps the first call's data
        rc = _noalloc(lib, la, S_new, *steps[step], outs[step], B, H, stream)
        assert rc == la.LA_OK, la.la_status_string(rc)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    # the same kernel with the allocating entry point's workspace: identical bits
    S_ref = S0.clone()
    for step in range(2):
        out_ref = la.la_decode_step(S_ref, *steps[step])
        torch.cuda.synchronize()
        assert torch.equal(outs[step], out_ref), f"step {step}: out differs"
    assert torch.equal(S_new, S_ref)
    assert la.la_get_device_status() == la.LA_OK


def test_noalloc_refuses_batches_beyond_scratch(env):
    torch, la = env
    B, H = la.LA_NOALLOC_MAX_HEADS // 64 + 1, 64
    lib = la.load_library()
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(6)]  # never dereferenced
    rc = lib.la_decode_step_noalloc(p[0], p[1], p[2], p[3], p[4], p[5], B, H, 128,
                                    la.LA_BF16, 1e-6, None)
    assert rc == la.LA_ERR_SCRATCH_LIMIT
