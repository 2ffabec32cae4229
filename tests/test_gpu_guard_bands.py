"""Guard bands around the outputs of the packed prefill, the input projection and the
softmax layer: each output is written into the middle of a larger buffer filled with a
sentinel, and the sentinel on both sides must be intact after the call (no store past
the last token, the last feature or a packed sequence's end).
"""
import pytest

pytestmark = pytest.mark.gpu

PAD = 4096          # elements on each side (a multiple of 8: keeps 16-byte alignment)
SENTINEL = -1234.0  # exactly representable in bf16


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    la.load_library()
    return torch, la


def _guarded(torch, shape, dtype=None):
    import math
    n = math.prod(shape)
    buf = torch.full((PAD + n + PAD,), SENTINEL, device="cuda",
                     dtype=dtype or torch.bfloat16)
    return buf, buf[PAD:PAD + n].view(shape)


def _intact(torch, buf):
    return bool(torch.all(buf[:PAD] == SENTINEL)) and bool(torch.all(buf[-PAD:] == SENTINEL))


def test_varlen_output_guard_bands(env):
    torch, la = env
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    lens = [130, 0, 77, 300]                       # every sequence ends mid-chunk
    T = sum(lens)
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    q, k, v, g = (t[0] for t in make_prefill_inputs(1, T, 4, 128, torch.bfloat16, 0.5, 81,
                                                      "cuda"))
    buf, out = _guarded(torch, (T, 4, 128))
    sbuf, S = _guarded(torch, (len(lens), 4, 128, 128), torch.float32)
    la.la_prefill_varlen(q, k, v, g, cu, out=out, kv_state_out=S)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    assert _intact(torch, buf) and _intact(torch, sbuf)
    assert not torch.any(out == SENTINEL)


def test_projection_output_guard_bands(env):
    torch, la = env
    from linear_attention_hybrid_fwd_b300.inputs import make_projection_inputs
    T, hidden, H = 300, 192, 2
    x, w = make_projection_inputs(T, hidden, H, 128, 82, "cuda")
    guarded = [_guarded(torch, (T, H, 128)) for _ in range(4)]
    la.la_qkvg_projection(x, w, H, activate=True, out=tuple(o for _, o in guarded))
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    for buf, o in guarded:
        assert _intact(torch, buf)
        assert not torch.any(o == SENTINEL)


def test_softmax_attention_output_guard_bands(env):
    torch, la = env
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    B, N, H = 2, 300, 3                            # a ragged last query tile
    q, k, v, _ = make_prefill_inputs(B, N, H, 128, torch.bfloat16, 1.0, 83, "cuda")
    buf, out = _guarded(torch, (B, N, H, 128))
    la.la_softmax_attention(q, k, v, out=out)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    assert _intact(torch, buf)
    assert not torch.any(out == SENTINEL)
