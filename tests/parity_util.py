"""Helpers shared by the GPU parity tests: host copies and error measures.

Tolerances (bf16 I/O with fp32 accumulation / fp32 I/O):
* post-norm output:  max|out - ref| <= 1e-2 * max|ref|   (fp32 I/O: 1e-4)
* pre-norm y, per token row of the [B*N, H*d] output:
      max|dy| / max|y_ref| <= 2e-2                        (fp32 I/O: 1e-4)
  and elementwise, against the sum of the magnitudes of the terms of each y:
      |dy| <= 1e-2 * Y_abs + 1e-6 * max(Y_abs)            (fp32 I/O: 1e-5)
  where Y_abs is the same recurrence on |q^|, |k^|, |v^| (and |S0|).  A single
  head's row can cancel (q^ . k^ sums 128 terms of both signs), so a bound relative
  to that row's own maximum is not met by any bf16-operand product; the elementwise
  bound is the standard forward-error bound of a dot product and holds in every row.
* state, elementwise: |dS| <= 1e-2 * S_abs + 1e-6 * max(S_abs)  (fp32 I/O: 1e-5), with
  S_abs = |S0| + sum_s |k^_s|^T |v^_s|: one bf16 rounding (unit roundoff 2^-8) of each
  MMA operand bounds a single product's relative error by 2^-7, so a sequence of a few
  tokens can reach ~0.8% of its largest element;
  and for sequences of >= 128 tokens, where the roundings average out, also
  max|dS| <= 5e-3 * max|S_ref|                              (fp32 I/O: 1e-5)
"""
import numpy as np

TOL = {
    "bf16": dict(out=1e-2, y_row=2e-2, y_elem=1e-2, state=5e-3),
    "f32": dict(out=1e-4, y_row=1e-4, y_elem=1e-5, state=1e-5),
}


def host64(t):
    """Exact fp64 copy of a CUDA tensor (bf16 and fp32 widen exactly)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_max_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def row_rel_err(got, ref, axes=(-1,)):
    """Worst over rows of max|d| / max|ref|; a row spans ``axes`` (default: the last
    axis, e.g. the d features of a decode head; ``(-2, -1)`` is a token's H*d row)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if tuple(axes) != (-1,):
        lead = got.shape[:len(got.shape) - len(axes)]
        got = got.reshape(lead + (-1,))
        ref = ref.reshape(lead + (-1,))
    num = np.abs(got - ref).max(-1)
    den = np.abs(ref).max(-1)
    den = np.where(den > 0, den, 1.0)
    return float((num / den).max())


def y_abs_bound(orc, q, k, v, S0=None):
    """The recurrence on |SiLU(q)|, |SiLU(k)|, |SiLU(v)| (and |S0|): for each y element,
    the sum of the magnitudes of the products that make it up."""
    qa, ka, va = (np.abs(orc.silu(x)) for x in (q, k, v))
    y, _ = orc.core(qa, ka, va, S0=None if S0 is None else np.abs(S0))
    return y


def state_abs_bound(orc, k, v, S0=None):
    """S_abs = |S0| + sum over tokens of |SiLU(k)|^T |SiLU(v)| per (b, h)."""
    ka, va = (np.abs(orc.silu(x)) for x in (k, v))
    _, S = orc.core(ka, ka, va, S0=None if S0 is None else np.abs(S0), want_y=False)
    return S


def state_ok(orc, got, ref, k, v, S0, dt):
    """The state checks above; returns (ok, message)."""
    tol = TOL[dt]
    n = np.asarray(k).shape[1]
    sabs = state_abs_bound(orc, k, v, S0)
    ok, worst = elem_bound_ok(got, ref, sabs, tol["y_elem"])
    if not ok:
        return False, f"state exceeds the elementwise bound by x{worst:.2f}"
    if n >= 128:
        e = rel_max_err(got, ref)
        if e > tol["state"]:
            return False, f"state rel err {e:.3e}"
    return True, ""


def elem_bound_ok(got, ref, yabs, rel):
    """|got - ref| <= rel * yabs + 1e-6 * max(yabs), elementwise; returns (ok, worst)."""
    got = np.asarray(got, np.float64)
    lim = rel * yabs + 1e-6 * float(np.abs(yabs).max())
    ratio = np.abs(got - ref) / lim
    return bool((ratio <= 1.0).all()), float(ratio.max())
