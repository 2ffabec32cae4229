"""Host-side checks of the C ABI (no GPU needed).

The library must load on a machine without a CUDA device, export every function that
``include/lightning_attn.h`` declares, and reject bad arguments on the host before
anything is launched (these calls never reach the CUDA runtime).
"""
import ctypes
import os
import re

import pytest

import linear_attention_hybrid_fwd_b300 as la
from linear_attention_hybrid_fwd_b300 import build as la_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    la_build.build()
    return la.load_library()


def _declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(?:int|int64_t|const char\s*\*|void)\s+(la_\w+)\s*\(", src):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ["la_prefill", "la_decode_step", "la_prefill_ex", "la_decode_step_ex",
                 "la_prefill_varlen", "la_prefill_varlen_ex", "la_qkvg_projection",
                 "la_softmax_attention",
                 "la_status_string", "la_get_device_status", "la_version", "la_launch_count",
                 "la_prefill_path"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    for s in range(7):
        assert la.la_status_string(s)
    assert "unknown" in la.la_status_string(99)
    assert la.la_version() >= 100


# Fake, 16-byte aligned, never-dereferenced device addresses: every call below must
# fail validation on the host, so no pointer is ever touched.
P = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
MIS = ctypes.c_void_p(0x10008)


def _prefill(lib, B=1, H=2, N=16, d=128, dtype=la.LA_BF16, eps=1e-6, flags=0, q=None,
             out=None, ptrs=None):
    p = list(ptrs or P)
    if q is not None:
        p[0] = q
    if out is not None:
        p[4] = out
    return lib.la_prefill_ex(p[0], p[1], p[2], p[3], p[4], p[5], None, None, B, H, N, d, dtype,
                             eps, flags, None)


@pytest.mark.parametrize("kw,want", [
    (dict(B=0), la.LA_ERR_INVALID_ARG),
    (dict(H=0), la.LA_ERR_INVALID_ARG),
    (dict(N=-1), la.LA_ERR_INVALID_ARG),
    (dict(d=0), la.LA_ERR_INVALID_ARG),
    (dict(d=64), la.LA_ERR_UNSUPPORTED),
    (dict(d=129), la.LA_ERR_UNSUPPORTED),
    (dict(dtype=7), la.LA_ERR_INVALID_ARG),
    (dict(eps=-1.0), la.LA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), la.LA_ERR_INVALID_ARG),
    (dict(flags=0x100), la.LA_ERR_INVALID_ARG),
    (dict(flags=8), la.LA_ERR_INVALID_ARG),
    (dict(flags=la.LA_FLAG_ACTIVATED, d=64), la.LA_ERR_UNSUPPORTED),  # flag itself accepted
    (dict(flags=la.LA_FLAG_SERIAL, d=64), la.LA_ERR_UNSUPPORTED),     # flag itself accepted
    (dict(q=ctypes.c_void_p(0)), la.LA_ERR_INVALID_ARG),
    (dict(q=MIS), la.LA_ERR_MISALIGNED),
    (dict(out=P[0]), la.LA_ERR_INVALID_ARG),           # out aliases q
    (dict(N=1 << 40), la.LA_ERR_INVALID_ARG),          # element count overflow guard
])
def test_prefill_rejects_on_host(lib, kw, want):
    assert _prefill(lib, **kw) == want


def test_prefill_entry_rejects_on_host(lib):
    assert lib.la_prefill(P[0], P[1], P[2], P[3], P[4], P[5], 1, 2, 16, 64) == \
        la.LA_ERR_UNSUPPORTED
    assert lib.la_prefill(None, P[1], P[2], P[3], P[4], P[5], 1, 2, 16, 128) == \
        la.LA_ERR_INVALID_ARG


@pytest.mark.parametrize("args,want", [
    (dict(B=0), la.LA_ERR_INVALID_ARG),
    (dict(H=-1), la.LA_ERR_INVALID_ARG),
    (dict(d=96), la.LA_ERR_UNSUPPORTED),
    (dict(dtype=3), la.LA_ERR_INVALID_ARG),
    (dict(state=ctypes.c_void_p(0)), la.LA_ERR_INVALID_ARG),
    (dict(state=MIS), la.LA_ERR_MISALIGNED),
    (dict(out=P[1]), la.LA_ERR_INVALID_ARG),           # out aliases q
])
def test_decode_rejects_on_host(lib, args, want):
    a = dict(B=2, H=2, d=128, dtype=la.LA_BF16, state=P[0], out=P[6])
    a.update(args)
    rc = lib.la_decode_step_ex(a["state"], P[1], P[2], P[3], P[4], a["out"], None, a["B"],
                               a["H"], a["d"], a["dtype"], 1e-6, None)
    assert rc == want


def test_decode_y_debug_must_not_overlap(lib):
    # the kernel writes fp32 y over [B][H][d]: it may not land on an input, out or the state
    for y in (P[0], P[1], P[4], P[6]):
        rc = lib.la_decode_step_ex(P[0], P[1], P[2], P[3], P[4], P[6], y, 2, 2, 128,
                                   la.LA_BF16, 1e-6, None)
        assert rc == la.LA_ERR_INVALID_ARG


def test_wrappers_make_the_tensors_device_current(monkeypatch):
    # the library launches on, and keeps its workspace for, the current device; the
    # wrappers switch to the tensors' device around the call when it is another one
    import torch
    calls = []

    class Guard:
        def __init__(self, dev):
            calls.append(("switch", dev.index))

        def __enter__(self):
            return self

        def __exit__(self, *exc):
            calls.append(("back",))

    class Dev:
        def __init__(self, index):
            self.index = index

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "device", Guard)
    with la._on_device(Dev(3)):
        calls.append(("call",))
    assert calls == [("switch", 3), ("call",), ("back",)]
    calls.clear()
    with la._on_device(Dev(0)):
        calls.append(("call",))
    assert calls == [("call",)]


def test_prefill_path_rejects_on_host(lib):
    assert lib.la_prefill_path(0, 1, 1, 128, la.LA_BF16, 0) == -la.LA_ERR_INVALID_ARG
    assert lib.la_prefill_path(1, 1, 1, 64, la.LA_BF16, 0) == -la.LA_ERR_UNSUPPORTED
    assert lib.la_prefill_path(1, 1, 1, 128, 9, 0) == -la.LA_ERR_INVALID_ARG
    assert lib.la_prefill_path(1, 1, 1, 128, la.LA_F32, 0) == 1   # fp32: CUDA-core kernel
    assert lib.la_prefill_path(1, 1, 1, 128, la.LA_BF16, la.LA_FLAG_SIMT) == 1
    assert lib.la_prefill_path(1, 1, 1, 128, la.LA_BF16, 8) == -la.LA_ERR_INVALID_ARG
    assert lib.la_prefill_path(1, 1, 1, 128, la.LA_F32, la.LA_FLAG_SERIAL) == 1


@pytest.mark.parametrize("cu,S,d,want", [
    ([0, 5, 3], 2, 128, la.LA_ERR_INVALID_ARG),     # decreasing offsets
    ([1, 5], 1, 128, la.LA_ERR_INVALID_ARG),        # does not start at 0
    ([0, 5], 0, 128, la.LA_ERR_INVALID_ARG),        # no sequence
    ([0, 5], 1, 64, la.LA_ERR_UNSUPPORTED),         # head size
])
def test_varlen_rejects_on_host(lib, cu, S, d, want):
    arr = (ctypes.c_int64 * len(cu))(*cu)
    rc = lib.la_prefill_varlen_ex(P[0], P[1], P[2], P[3], P[4], P[5], None, None, arr, S, 2, d,
                                  la.LA_BF16, 1e-6, 0, None)
    assert rc == want
    assert lib.la_prefill_varlen_ex(P[0], P[1], P[2], P[3], P[4], P[5], None, None, None, 1, 2,
                                    128, la.LA_BF16, 1e-6, 0, None) == la.LA_ERR_INVALID_ARG


def test_decode_entry_rejects_on_host(lib):
    assert lib.la_decode_step(P[0], P[1], P[2], P[3], P[4], P[5], 1, 1, 32) == \
        la.LA_ERR_UNSUPPORTED


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """The binding has no other implementation: without the .so it raises."""
    monkeypatch.setattr(la, "_lib", None)
    monkeypatch.setattr(la, "_LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        la.load_library()


def test_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "linear_attention_hybrid_fwd_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "la_oracle" not in src, f


def _proj(lib, T=16, hidden=64, H=2, d=128, flags=la.LA_PROJ_SILU, x=None, q=None):
    return lib.la_qkvg_projection(x if x is not None else P[0], P[1],
                                  q if q is not None else P[2], P[3], P[4], P[5], T, hidden,
                                  H, d, flags, None)


@pytest.mark.parametrize("kw,want", [
    (dict(T=-1), la.LA_ERR_INVALID_ARG),
    (dict(hidden=0), la.LA_ERR_INVALID_ARG),
    (dict(H=0), la.LA_ERR_INVALID_ARG),
    (dict(d=64), la.LA_ERR_UNSUPPORTED),
    (dict(H=1), la.LA_ERR_UNSUPPORTED),                # H*d not a multiple of 256
    (dict(hidden=12), la.LA_ERR_UNSUPPORTED),          # rows not 16-byte strided
    (dict(flags=2), la.LA_ERR_INVALID_ARG),
    (dict(x=ctypes.c_void_p(0)), la.LA_ERR_INVALID_ARG),
    (dict(x=MIS), la.LA_ERR_MISALIGNED),
    (dict(q=P[0]), la.LA_ERR_INVALID_ARG),             # q aliases x
    (dict(q=P[3]), la.LA_ERR_INVALID_ARG),             # q aliases k
])
def test_projection_rejects_on_host(lib, kw, want):
    assert _proj(lib, **kw) == want


def test_projection_empty_batch_launches_nothing(lib):
    n0 = lib.la_launch_count()
    assert _proj(lib, T=0) == la.LA_OK
    assert lib.la_launch_count() == n0


def _attn(lib, B=1, H=2, N=16, d=128, base=1e7, q=None, out=None):
    return lib.la_softmax_attention(q if q is not None else P[0], P[1], P[2],
                                    out if out is not None else P[3], B, H, N, d, base, None)


@pytest.mark.parametrize("kw,want", [
    (dict(B=0), la.LA_ERR_INVALID_ARG),
    (dict(H=-1), la.LA_ERR_INVALID_ARG),
    (dict(N=-1), la.LA_ERR_INVALID_ARG),
    (dict(d=64), la.LA_ERR_UNSUPPORTED),
    (dict(base=1.0), la.LA_ERR_INVALID_ARG),
    (dict(base=float("inf")), la.LA_ERR_INVALID_ARG),
    (dict(base=float("nan")), la.LA_ERR_INVALID_ARG),
    (dict(q=ctypes.c_void_p(0)), la.LA_ERR_INVALID_ARG),
    (dict(q=MIS), la.LA_ERR_MISALIGNED),
    (dict(out=P[1]), la.LA_ERR_INVALID_ARG),           # out aliases k
    (dict(N=(1 << 30) + 1), la.LA_ERR_UNSUPPORTED),
])
def test_softmax_attention_rejects_on_host(lib, kw, want):
    assert _attn(lib, **kw) == want


def test_softmax_attention_empty_launches_nothing(lib):
    n0 = lib.la_launch_count()
    assert _attn(lib, N=0) == la.LA_OK
    assert lib.la_launch_count() == n0
