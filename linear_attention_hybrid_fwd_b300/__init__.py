"""Lightning Attention forward on B300 (sm_103a): a thin ctypes binding.

This module only marshals arguments to ``liblightning_attn.so`` (the C ABI declared in
``include/lightning_attn.h``): torch tensors become device pointers, torch's current
CUDA stream becomes the ``cudaStream_t``.  Every step of the computation runs in the
library's CUDA kernels.  There is no other implementation: if the library is missing
or no CUDA device is present, the calls raise.

Functions carry the C names:

* ``la_prefill(q, k, v, g, ...)``       -- prefill of ``[B, N, H, d]`` inputs
* ``la_prefill_varlen(q, k, v, g, cu_seqlens, ...)`` -- packed sequences of any lengths
* ``la_decode_step(kv_state, q, ...)``  -- one token per sequence, ``[B, H, d]`` inputs
* ``la_decode_step_noalloc``           -- the same step with the library's fixed scratch,
                                          for callers that cannot let it allocate
* ``la_state_pass(k, v, ...)``         -- the state after a run of tokens, no outputs
* ``la_state_sum(parts, base)``        -- fixed-order sum of states (sharded prefill)
* ``la_prefill_path``                  -- which prefill kernel serves a shape
* ``la_status_string``, ``la_get_device_status``, ``la_version``, ``la_launch_count``
"""
from __future__ import annotations

import contextlib
import ctypes
import os

__all__ = ["la_prefill", "la_prefill_varlen", "la_decode_step", "la_decode_step_noalloc",
           "la_state_pass", "la_state_sum",
           "la_qkvg_projection", "la_softmax_attention", "la_status_string", "la_get_device_status", "la_version",
           "la_launch_count", "la_prefill_path", "LaError", "library_path", "load_library",
           "LA_BF16", "LA_F32", "LA_FLAG_SIMT", "LA_FLAG_ACTIVATED", "LA_FLAG_SERIAL",
           "LA_PROJ_SILU"]

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_MISALIGNED = 0, 1, 2, 3
LA_ERR_CUDA, LA_ERR_NOMEM, LA_ERR_TIMEOUT, LA_ERR_SCRATCH_LIMIT = 4, 5, 6, 7
LA_NOALLOC_MAX_HEADS = 16384
LA_BF16, LA_F32 = 0, 1
LA_FLAG_SIMT = 1
LA_FLAG_ACTIVATED = 2
LA_FLAG_SERIAL = 4
LA_PROJ_SILU = 1

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "liblightning_attn.so")
_lib = None


class LaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {la_status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load ``liblightning_attn.so`` (built in-tree by ``build.py``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: run `python -m linear_attention_hybrid_fwd_b300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, fp, i32, i64, f32, u32 = (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                  ctypes.c_int64, ctypes.c_float, ctypes.c_uint)
    lib.la_prefill.argtypes = [vp, vp, vp, vp, vp, fp, i32, i32, i64, i32]
    lib.la_prefill.restype = i32
    lib.la_prefill_ex.argtypes = [vp, vp, vp, vp, vp, fp, fp, fp, i32, i32, i64, i32, i32, f32,
                                  u32, vp]
    lib.la_prefill_ex.restype = i32
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.la_prefill_varlen_ex.argtypes = [vp, vp, vp, vp, vp, fp, fp, fp, i64p, i32, i32, i32, i32,
                                         f32, u32, vp]
    lib.la_prefill_varlen_ex.restype = i32
    lib.la_prefill_varlen.argtypes = [vp, vp, vp, vp, vp, fp, i64p, i32, i32, i32]
    lib.la_prefill_varlen.restype = i32
    lib.la_decode_step.argtypes = [fp, vp, vp, vp, vp, vp, i32, i32, i32]
    lib.la_decode_step.restype = i32
    lib.la_decode_step_ex.argtypes = [fp, vp, vp, vp, vp, vp, fp, i32, i32, i32, i32, f32, vp]
    lib.la_decode_step_ex.restype = i32
    lib.la_decode_step_noalloc.argtypes = [fp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, vp]
    lib.la_decode_step_noalloc.restype = i32
    lib.la_status_string.argtypes = [i32]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_get_device_status.argtypes = [vp]
    lib.la_get_device_status.restype = i32
    lib.la_version.argtypes = []
    lib.la_version.restype = i32
    lib.la_prefill_path.argtypes = [i32, i32, i64, i32, i32, u32]
    lib.la_prefill_path.restype = i32
    lib.la_qkvg_projection.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, u32, vp]
    lib.la_qkvg_projection.restype = i32
    lib.la_softmax_attention.argtypes = [vp, vp, vp, vp, i32, i32, i64, i32, ctypes.c_double,
                                         vp]
    lib.la_softmax_attention.restype = i32
    lib.la_state_pass.argtypes = [vp, vp, fp, fp, i32, i32, i64, i32, i32, u32, vp]
    lib.la_state_pass.restype = i32
    lib.la_state_sum.argtypes = [fp, i32, fp, fp, i64, vp]
    lib.la_state_sum.restype = i32
    lib.la_launch_count.argtypes = []
    lib.la_launch_count.restype = ctypes.c_int64
    _lib = lib
    return lib


def la_status_string(status: int) -> str:
    return load_library().la_status_string(int(status)).decode()


def la_version() -> int:
    return load_library().la_version()


def la_prefill_path(B: int, H: int, N: int, d: int = 128, dtype: int = LA_BF16,
                    simt: bool = False, serial: bool = False) -> int:
    """0 if the tensor-core prefill kernel serves this shape, 1 for the CUDA-core one,
    2 for the tensor-core kernel in the segment-parallel mode."""
    return load_library().la_prefill_path(B, H, N, d, dtype, _prefill_flags(simt, False, serial))


def la_launch_count() -> int:
    return load_library().la_launch_count()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def la_get_device_status(stream=None) -> int:
    return load_library().la_get_device_status(_stream_handle(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return LA_BF16
    if t.dtype == torch.float32:
        return LA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: expected bfloat16 or float32")


def _check(ts, names):
    """Checks that every given tensor is a contiguous CUDA tensor on one device; returns
    that device."""
    import torch
    dev = None
    for t, n in zip(ts, names):
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{n} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{n} is on {t.device}, expected {dev}")
    return dev


@contextlib.contextmanager
def _on_device(dev):
    """Makes the tensors' device current for the library call: the library launches on,
    and keeps its workspace for, the current device, and the stream handle is taken
    from the current device's current stream."""
    import torch
    if dev is None or dev.index is None or dev.index == torch.cuda.current_device():
        yield
    else:
        with torch.cuda.device(dev):
            yield


def _prefill_flags(simt, activated, serial=False):
    return ((LA_FLAG_SIMT if simt else 0) | (LA_FLAG_ACTIVATED if activated else 0)
            | (LA_FLAG_SERIAL if serial else 0))


def la_prefill(q, k, v, g, out=None, kv_state_out=None, kv_state_in=None, y_debug=None,
               eps: float = 1e-6, simt: bool = False, want_state: bool = True, stream=None,
               activated: bool = False, serial: bool = False):
    """Prefill. ``q, k, v, g``: ``[B, N, H, d]`` (bf16 or fp32, contiguous, CUDA).

    Returns ``(out, kv_state_out)``; ``kv_state_out`` is ``[B, H, d, d]`` fp32 (``None``
    when ``want_state`` is False and none was passed).  ``kv_state_in`` continues a
    sequence from a previous state; ``y_debug`` (fp32 ``[B, N, H, d]``) receives the
    pre-norm output.  ``simt`` selects the CUDA-core kernel.  ``activated``: q, k, v
    are already SiLU-activated (``la_qkvg_projection(..., activate=True)``).  ``serial``
    keeps one chunk chain per head where the segment-parallel mode would run.
    """
    import torch
    B, N, H, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if kv_state_out is None and want_state:
        kv_state_out = torch.empty((B, H, d, d), device=q.device, dtype=torch.float32)
    _check([q, k, v, g, out, kv_state_out, kv_state_in, y_debug],
           ["q", "k", "v", "g", "out", "kv_state_out", "kv_state_in", "y_debug"])
    for t, n in ((k, "k"), (v, "v"), (g, "g"), (out, "out")):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    for t, n in ((kv_state_out, "kv_state_out"), (kv_state_in, "kv_state_in")):
        if t is not None and (t.shape != (B, H, d, d) or t.dtype != torch.float32):
            raise ValueError(f"{n} must be float32 [B, H, d, d]")
    if y_debug is not None and (y_debug.shape != q.shape or y_debug.dtype != torch.float32):
        raise ValueError("y_debug must be float32 [B, N, H, d]")
    with _on_device(q.device):
        rc = load_library().la_prefill_ex(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out), _ptr(kv_state_out),
            _ptr(kv_state_in), _ptr(y_debug), B, H, N, d, _dtype_code(q), float(eps),
            _prefill_flags(simt, activated, serial), _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_prefill")
    return out, kv_state_out


def la_prefill_varlen(q, k, v, g, cu_seqlens, out=None, kv_state_out=None, kv_state_in=None,
                      y_debug=None, eps: float = 1e-6, simt: bool = False, want_state: bool = True,
                      stream=None, activated: bool = False):
    """Packed prefill: ``q, k, v, g`` are ``[T, H, d]`` (bf16 or fp32, contiguous, CUDA),
    sequence ``b`` is rows ``cu_seqlens[b]:cu_seqlens[b+1]`` (``cu_seqlens``: host ints,
    ``num_seqs + 1`` of them, starting at 0).  Returns ``(out, kv_state_out)`` with
    ``kv_state_out`` ``[num_seqs, H, d, d]`` fp32."""
    import torch
    T, H, d = q.shape
    cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                           else cu_seqlens)]
    S = len(cu) - 1
    if S < 1:
        raise ValueError("cu_seqlens needs at least two entries")
    if cu[-1] != T:
        raise ValueError(f"cu_seqlens ends at {cu[-1]}, q has {T} tokens")
    if out is None:
        out = torch.empty_like(q)
    if kv_state_out is None and want_state:
        kv_state_out = torch.empty((S, H, d, d), device=q.device, dtype=torch.float32)
    _check([q, k, v, g, out, kv_state_out, kv_state_in, y_debug],
           ["q", "k", "v", "g", "out", "kv_state_out", "kv_state_in", "y_debug"])
    for t, n in ((k, "k"), (v, "v"), (g, "g"), (out, "out")):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    for t, n in ((kv_state_out, "kv_state_out"), (kv_state_in, "kv_state_in")):
        if t is not None and (tuple(t.shape) != (S, H, d, d) or t.dtype != torch.float32):
            raise ValueError(f"{n} must be float32 [num_seqs, H, d, d]")
    if y_debug is not None and (y_debug.shape != q.shape or y_debug.dtype != torch.float32):
        raise ValueError("y_debug must be float32 [T, H, d]")
    cu_arr = (ctypes.c_int64 * (S + 1))(*cu)
    with _on_device(q.device):
        rc = load_library().la_prefill_varlen_ex(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out), _ptr(kv_state_out),
            _ptr(kv_state_in), _ptr(y_debug), cu_arr, S, H, d, _dtype_code(q), float(eps),
            _prefill_flags(simt, activated), _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_prefill_varlen")
    return out, kv_state_out


def la_qkvg_projection(x, w, H: int, d: int = 128, activate: bool = True, out=None,
                       stream=None):
    """Input projection on tensor cores: ``x`` ``[T, hidden]`` bf16, ``w`` ``[4*H*d,
    hidden]`` bf16 (rows: q, k, v, g features).  Returns ``(q, k, v, g)``, each bf16
    ``[T, H, d]``; q, k, v are SiLU-activated when ``activate`` (feed them to
    ``la_prefill(..., activated=True)``), otherwise raw.  ``out``: optional tuple of four
    preallocated outputs."""
    import torch
    if x.dim() != 2 or w.dim() != 2:
        raise ValueError("x must be [T, hidden] and w [4*H*d, hidden]")
    T, hidden = x.shape
    if tuple(w.shape) != (4 * H * d, hidden):
        raise ValueError(f"w must be [{4 * H * d}, {hidden}], got {tuple(w.shape)}")
    if out is None:
        out = tuple(torch.empty((T, H, d), device=x.device, dtype=x.dtype) for _ in range(4))
    _check([x, w, *out], ["x", "w", "q", "k", "v", "g"])
    for t in (x, w, *out):
        if t.dtype != torch.bfloat16:
            raise ValueError("la_qkvg_projection takes and returns bf16 tensors")
    for t in out:
        if tuple(t.shape) != (T, H, d):
            raise ValueError(f"outputs must be [{T}, {H}, {d}]")
    with _on_device(x.device):
        rc = load_library().la_qkvg_projection(
            _ptr(x), _ptr(w), *(_ptr(t) for t in out), T, hidden, H, d,
            LA_PROJ_SILU if activate else 0, _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_qkvg_projection")
    return out


def la_softmax_attention(q, k, v, out=None, rope_base: float = 1.0e7, stream=None):
    """The softmax layer: RoPE on the first half of each head's features, then causal
    softmax attention.  ``q, k, v``: bf16 ``[B, N, H, 128]`` (contiguous, CUDA).
    Returns ``out`` of the same shape."""
    import torch
    B, N, H, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check([q, k, v, out], ["q", "k", "v", "out"])
    for t, n in ((k, "k"), (v, "v"), (out, "out")):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    if q.dtype != torch.bfloat16:
        raise ValueError("la_softmax_attention takes bf16 tensors")
    with _on_device(q.device):
        rc = load_library().la_softmax_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H,
                                                 N, d, float(rope_base), _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_softmax_attention")
    return out


def la_decode_step(kv_state, q, k, v, g, out=None, y_debug=None, eps: float = 1e-6,
                   stream=None):
    """One decode step. ``kv_state`` ``[B, H, d, d]`` fp32 is updated in place;
    ``q, k, v, g`` are ``[B, H, d]``.  Returns ``out`` (``[B, H, d]``, dtype of q)."""
    import torch
    B, H, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check([kv_state, q, k, v, g, out, y_debug],
           ["kv_state", "q", "k", "v", "g", "out", "y_debug"])
    for t, n in ((k, "k"), (v, "v"), (g, "g"), (out, "out")):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    if kv_state.shape != (B, H, d, d) or kv_state.dtype != torch.float32:
        raise ValueError("kv_state must be float32 [B, H, d, d]")
    with _on_device(q.device):
        rc = load_library().la_decode_step_ex(
            _ptr(kv_state), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out), _ptr(y_debug), B,
            H, d, _dtype_code(q), float(eps), _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_decode_step")
    return out


def la_decode_step_noalloc(kv_state, q, k, v, g, out, eps: float = 1e-6, stream=None):
    """``la_decode_step`` for callers that cannot let the library allocate device
    memory: the kernels' scratch is a fixed array inside the library (up to
    ``LA_NOALLOC_MAX_HEADS`` = B*H heads).  ``out`` must be given, so this wrapper
    allocates nothing either.  Calls on one device share the scratch: order calls
    that could overlap on the GPU."""
    B, H, d = q.shape
    _check([kv_state, q, k, v, g, out], ["kv_state", "q", "k", "v", "g", "out"])
    for t, n in ((k, "k"), (v, "v"), (g, "g"), (out, "out")):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{n} must match q in shape and dtype")
    if tuple(kv_state.shape) != (B, H, d, d) or kv_state.dtype != _float32():
        raise ValueError("kv_state must be float32 [B, H, d, d]")
    with _on_device(q.device):
        rc = load_library().la_decode_step_noalloc(
            _ptr(kv_state), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(out), B, H, d,
            _dtype_code(q), float(eps), _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_decode_step_noalloc")
    return out


def la_state_pass(k, v, kv_state_out=None, kv_state_in=None, activated: bool = False,
                  stream=None):
    """State after the tokens of ``k, v`` (bf16 ``[B, N, H, d]``) without computing
    outputs: ``kv_state_in + SiLU(K)^T SiLU(V)`` per (sequence, head), fp32
    ``[B, H, d, d]``.  ``activated``: k and v are already SiLU-activated."""
    import torch
    B, N, H, d = k.shape
    if kv_state_out is None:
        kv_state_out = torch.empty((B, H, d, d), device=k.device, dtype=torch.float32)
    _check([k, v, kv_state_out, kv_state_in], ["k", "v", "kv_state_out", "kv_state_in"])
    if v.shape != k.shape or v.dtype != k.dtype:
        raise ValueError("v must match k in shape and dtype")
    for t, n in ((kv_state_out, "kv_state_out"), (kv_state_in, "kv_state_in")):
        if t is not None and (tuple(t.shape) != (B, H, d, d) or t.dtype != torch.float32):
            raise ValueError(f"{n} must be float32 [B, H, d, d]")
    with _on_device(k.device):
        rc = load_library().la_state_pass(
            _ptr(k), _ptr(v), _ptr(kv_state_out), _ptr(kv_state_in), B, H, N, d,
            _dtype_code(k), LA_FLAG_ACTIVATED if activated else 0, _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_state_pass")
    return kv_state_out


def la_state_sum(parts, base=None, out=None, stream=None):
    """``base + parts[0] + ... + parts[-1]`` added in that order (fp32 arrays; ``parts``
    is ``[count, ...]``, ``base`` and ``out`` shaped like ``parts[0]``)."""
    import torch
    shape = tuple(parts.shape[1:])
    if out is None:
        out = torch.empty(shape, device=parts.device, dtype=torch.float32)
    _check([parts, base, out], ["parts", "base", "out"])
    for t, n in ((parts, "parts"), (base, "base"), (out, "out")):
        if t is not None and t.dtype != torch.float32:
            raise ValueError(f"{n} must be float32")
    for t, n in ((base, "base"), (out, "out")):
        if t is not None and tuple(t.shape) != shape:
            raise ValueError(f"{n} must have the shape of parts[0]")
    with _on_device(parts.device):
        rc = load_library().la_state_sum(_ptr(parts), int(parts.shape[0]), _ptr(base),
                                         _ptr(out), out.numel(), _stream_handle(stream))
    if rc != LA_OK:
        raise LaError(rc, "la_state_sum")
    return out


def _float32():
    import torch
    return torch.float32
