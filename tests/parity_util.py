"""Helpers shared by the GPU parity tests: host copies and error measures.

Tolerances (bf16 I/O with fp32 accumulation / fp32 I/O):
* post-norm output:  max|out - ref| <= 1e-2 * max|ref|   (fp32 I/O: 1e-4)
* pre-norm y, per (b, t, h) row of d features: max|dy| / max|y_ref| <= 2e-2 (fp32: 1e-4)
* state: max|dS| <= 5e-3 * max|S_ref|                     (fp32 I/O: 1e-5)
"""
import numpy as np

TOL = {
    "bf16": dict(out=1e-2, y_row=2e-2, state=5e-3),
    "f32": dict(out=1e-4, y_row=1e-4, state=1e-5),
}


def host64(t):
    """Exact fp64 copy of a CUDA tensor (bf16 and fp32 widen exactly)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_max_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def row_rel_err(got, ref):
    """Worst over rows (last axis = the d features of one head) of max|d| / max|ref|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.abs(got - ref).max(-1)
    den = np.abs(ref).max(-1)
    den = np.where(den > 0, den, 1.0)
    return float((num / den).max())
