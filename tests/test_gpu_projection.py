"""GPU parity of the input projection (la_qkvg_projection) and of the prefill fed by it.

The projection is checked element by element against the fp64 oracle
(oracle/projection.py) on the exact bf16 bits the GPU read.  Bound per element:

    |got - ref| <= 2^-8 |ref| + 2^-11 |raw| + 2^-16 sum_i |x_i w_i|

* 2^-8 |ref|: the one RNE rounding to bf16 (half an ulp of an 8-bit significand);
* 2^-11 |raw|: SiLU as raw/2 (1 + tanh(raw/2)) with the hardware tanh approximation
  (relative error about 2^-11), which is absolute in raw where SiLU is small;
* 2^-16 sum |x_i w_i|: fp32 accumulation of up to 6144 exact bf16 products (about
  256 unit roundoffs of the magnitude sum, far above what a blocked sum reaches).
The layer fed by activated projections keeps the layer's own tolerances.
"""
import numpy as np
import pytest

from parity_util import TOL, host64, rel_max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    la.load_library()
    from oracle import projection
    return torch, la, oracle_mod, projection


def _xw(torch, T, hidden, H, d, seed, wscale=None):
    from linear_attention_hybrid_fwd_b300.inputs import make_projection_inputs
    return make_projection_inputs(T, hidden, H, d, seed, "cuda", wscale)


def _check_proj(prj, got, x64, w64, H, d, activate, rows=None):
    """got: the four GPU outputs [T, H, d] (or their sampled rows)."""
    ref = prj.project(x64, w64, H, d, activate=activate)
    raw = prj.project(x64, w64, H, d, activate=False)
    mag = prj.project(np.abs(x64), np.abs(w64), H, d, activate=False)
    for s, name in enumerate("qkvg"):
        g = host64(got[s]) if rows is None else host64(got[s][rows])
        bound = 2.0 ** -8 * np.abs(ref[s]) + 2.0 ** -11 * np.abs(raw[s]) + 2.0 ** -16 * mag[s]
        err = np.abs(g - ref[s])
        worst = float((err / np.maximum(bound, 1e-300)).max())
        assert worst <= 1.0, f"{name}: error {worst:.2f}x the bound"


@pytest.mark.parametrize("T,hidden,H", [(1, 64, 2), (130, 200, 2), (300, 512, 4), (513, 128, 2)])
@pytest.mark.parametrize("activate", [True, False])
def test_projection_small(env, T, hidden, H, activate):
    torch, la, _, prj = env
    x, w = _xw(torch, T, hidden, H, 128, 11 + T + hidden)
    out = la.la_qkvg_projection(x, w, H, activate=activate)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    _check_proj(prj, out, host64(x), host64(w), H, 128, activate)


def test_projection_gate_is_never_activated(env):
    torch, la, _, _ = env
    x, w = _xw(torch, 257, 192, 2, 128, 5)
    a = la.la_qkvg_projection(x, w, 2, activate=True)
    b = la.la_qkvg_projection(x, w, 2, activate=False)
    torch.cuda.synchronize()
    assert torch.equal(a[3], b[3])
    assert not torch.equal(a[0], b[0])


def test_projection_full_size_sampled_rows(env):
    """T = 8192 tokens, hidden 6144, H = 64 x 128 (the 8K prefill's projection), the
    launch bench.py times; 48 seeded rows (first and last tile included) checked in
    full against the oracle."""
    torch, la, _, prj = env
    from linear_attention_hybrid_fwd_b300.inputs import WORKLOADS
    wl = WORKLOADS["proj_8k"]
    x, w = _xw(torch, wl.N, wl.hidden, wl.H, wl.d, wl.seed)
    out = la.la_qkvg_projection(x, w, wl.H, activate=True)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    rng = np.random.default_rng(wl.seed)
    rows = sorted(set([0, 127, 128, wl.N - 1] + [int(r) for r in rng.integers(0, wl.N, 44)]))
    rows_t = torch.tensor(rows, device="cuda")
    _check_proj(prj, out, host64(x[rows_t]), host64(w), wl.H, wl.d, True, rows=rows_t)


@pytest.mark.parametrize("simt", [False, True])
def test_projection_feeds_prefill(env, simt):
    """x -> la_qkvg_projection(activate) -> la_prefill(activated=True) against the
    oracle layer on the fp64 projection of the same x and W; and against the oracle
    core on the exact activated bits the prefill read."""
    torch, la, orc, prj = env
    T, hidden, H = 300, 256, 2
    x, w = _xw(torch, T, hidden, H, 128, 21)
    q, k, v, g = la.la_qkvg_projection(x, w, H, activate=True)
    out, S = la.la_prefill(*(t.unsqueeze(0) for t in (q, k, v, g)), activated=True, simt=simt)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    raw = [o[None] for o in prj.project(host64(x), host64(w), H, 128, activate=False)]
    ref_out, _, ref_S = orc.prefill(*raw)
    assert rel_max_err(host64(out), ref_out) <= TOL["bf16"]["out"]
    assert rel_max_err(host64(S), ref_S) <= 2 * TOL["bf16"]["state"]
    # the same activated bits through the oracle's core: the kernel's own error only
    y, S_core = orc.core(*(host64(t)[None] for t in (q, k, v)))
    ref2 = orc.rmsnorm_gate(y, host64(g)[None])
    assert rel_max_err(host64(out), ref2) <= TOL["bf16"]["out"]
    assert rel_max_err(host64(S), S_core) <= TOL["bf16"]["state"]


def test_activated_flag_equals_raw_path_on_activated_bits(env):
    """la_prefill(activated=True) on q^ equals the oracle core on q^, and the varlen
    entry point takes the flag too."""
    torch, la, orc, _ = env
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    q, k, v, g = make_prefill_inputs(1, 700, 4, 128, torch.bfloat16, 0.5, 33, "cuda")
    qa, ka, va = (torch.nn.functional.silu(t.float()).to(torch.bfloat16) for t in (q, k, v))
    out, S = la.la_prefill(qa, ka, va, g, activated=True)
    cu = [0, 250, 250, 700]
    out_v, S_v = la.la_prefill_varlen(*(t[0] for t in (qa, ka, va, g)), cu, activated=True)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    y, S_ref = orc.core(*(host64(t) for t in (qa, ka, va)))
    ref = orc.rmsnorm_gate(y, host64(g))
    assert rel_max_err(host64(out), ref) <= TOL["bf16"]["out"]
    assert rel_max_err(host64(S), S_ref) <= TOL["bf16"]["state"]
    for b, (r0, r1) in enumerate(zip(cu[:-1], cu[1:])):
        if r1 == r0:
            assert torch.count_nonzero(S_v[b]) == 0
            continue
        y, S_ref = orc.core(*(host64(t[:, r0:r1]) for t in (qa, ka, va)))
        ref = orc.rmsnorm_gate(y, host64(g[:, r0:r1]))
        assert rel_max_err(host64(out_v[r0:r1]), ref[0]) <= TOL["bf16"]["out"]
        assert rel_max_err(host64(S_v[b:b + 1]), S_ref) <= TOL["bf16"]["state"]
