"""GPU parity of la_prefill against the fp64 oracle (same seeded input bits).

Covers the tensor-core kernel (bf16 default) and the CUDA-core kernel (fp32 I/O and
``LA_FLAG_SIMT``), shapes that span several 128-token chunks with ragged tails, the
64-head 8K-token workload in full, the 128K-token workload on sampled windows plus
the final state, and the edge cases (N = 0, N = 1, continuation from a state,
determinism, guard bands).
"""
import numpy as np
import pytest

from parity_util import (TOL, elem_bound_ok, host64, rel_max_err, row_rel_err, state_ok,
                         y_abs_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from linear_attention_hybrid_fwd_b300 import build as la_build
    la_build.build()
    import linear_attention_hybrid_fwd_b300 as la
    la.load_library()
    return torch, la, oracle_mod


def _inputs(torch, B, N, H, dtype, scale, seed):
    from linear_attention_hybrid_fwd_b300.inputs import make_prefill_inputs
    return make_prefill_inputs(B, N, H, 128, dtype, scale, seed, "cuda")


def _check_head_rows(y, ref_y, yabs, lim):
    """The error of each head's d-row of y relative to that row's own maximum.  A row can
    exceed ``lim`` only by cancellation: its reference is then small against the
    magnitudes that make it up (max|y_ref| < 0.05 max Y_abs of the row)."""
    num = np.abs(y - ref_y).max(-1)
    den = np.abs(ref_y).max(-1)
    err = num / np.where(den > 0, den, 1.0)
    big = err > lim
    cancel = den < 0.05 * np.abs(yabs).max(-1)
    print(f"per-head y rows: worst {err.max():.3e}, {int(big.sum())} of {err.size} above "
          f"{lim:g}, all of them cancellation rows: {bool(cancel[big].all())}")
    assert cancel[big].all(), "a head row above the bound is not a cancellation row"


def _check_prefill(env, B, N, H, dt, scale, seed, simt, S0=False, per_head=False):
    torch, la, orc = env
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    q, k, v, g = _inputs(torch, B, N, H, dtype, scale, seed)
    S_in = None
    if S0:
        gen = torch.Generator(device="cuda").manual_seed(seed + 99)
        S_in = torch.randn((B, H, 128, 128), generator=gen, device="cuda") * 0.5
    y = torch.empty((B, N, H, 128), device="cuda", dtype=torch.float32)
    out, S = la.la_prefill(q, k, v, g, kv_state_in=S_in, y_debug=y, simt=simt)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    ref_out, ref_y, ref_S = orc.prefill(host64(q), host64(k), host64(v), host64(g),
                                        S0=None if S_in is None else host64(S_in))
    tol = TOL[dt]
    e_out = rel_max_err(host64(out), ref_out)
    e_y = row_rel_err(host64(y), ref_y, axes=(-2, -1))
    e_S = rel_max_err(host64(S), ref_S)
    yabs = y_abs_bound(orc, host64(q), host64(k), host64(v),
                       None if S_in is None else host64(S_in))
    ok_elem, worst = elem_bound_ok(host64(y), ref_y, yabs, tol["y_elem"])
    assert e_out <= tol["out"], f"out rel err {e_out:.3e}"
    assert e_y <= tol["y_row"], f"y token-row err {e_y:.3e}"
    assert ok_elem, f"y exceeds the elementwise bound by x{worst:.2f}"
    if per_head:
        _check_head_rows(host64(y), ref_y, yabs, tol["y_row"])
    ok_S, msg = state_ok(orc, host64(S), ref_S, host64(k), host64(v),
                         None if S_in is None else host64(S_in), dt)
    assert ok_S, msg
    assert np.isfinite(host64(out)).all()
    return e_out, e_y, e_S


def test_tensor_core_path_selected(env):
    """bf16 at the 64-head shapes runs the tensor-core kernel; fp32 or the flag the
    CUDA-core one."""
    torch, la, _ = env
    for N in (1, 300, 8192, 131072, 1 << 20):
        assert la.la_prefill_path(1, 64, N) == 0, N
    assert la.la_prefill_path(1, 64, 8192, simt=True) == 1
    assert la.la_prefill_path(1, 64, 8192, dtype=la.LA_F32) == 1
    # one long sequence with few heads: the segment-parallel mode, unless asked not to
    assert la.la_prefill_path(1, 8, 40000) == 2
    assert la.la_prefill_path(1, 8, 40000, serial=True) == 0
    assert la.la_prefill_path(2, 8, 40000) == 0       # only B == 1 is cut
    assert la.la_prefill_path(1, 8, 16000) == 0       # under two segments of 64 chunks
    assert la.la_prefill_path(1, 37, 1 << 20) == 0    # 2 x 37 head pairs do not fit
    assert la.la_prefill_path(1, 36, 1 << 20) == 2


def test_tiny_f32_workload(env):
    """fp32 I/O: B1 H1 N512 d128, N(0,1) seed 0, norm over the d features; tol 1e-4."""
    _check_prefill(env, 1, 512, 1, "f32", 1.0, 0, simt=True)


@pytest.mark.parametrize("simt", [False, True])
@pytest.mark.parametrize("B,N,H", [(1, 1, 1), (1, 127, 2), (2, 300, 4), (1, 1000, 3),
                                   (3, 129, 8), (1, 257, 64)])
def test_bf16_shapes(env, B, N, H, simt):
    _check_prefill(env, B, N, H, "bf16", 0.5, 11 + N + H, simt=simt)


@pytest.mark.parametrize("simt", [False, True])
def test_bf16_with_initial_state(env, simt):
    _check_prefill(env, 2, 333, 4, "bf16", 0.5, 21, simt=simt, S0=True)


def test_f32_shapes(env):
    _check_prefill(env, 2, 200, 3, "f32", 1.0, 31, simt=True, S0=True)


def test_tensor_core_head_limit(env):
    """The tensor-core kernel keeps every head pair and at least one reducer pair resident:
    at the largest head count it takes (73 two-CTA clusters on a 148-SM B300) it matches
    the oracle; one head more, bf16 without LA_FLAG_SIMT is refused (no silent switch of
    kernel), and with LA_FLAG_SIMT the CUDA-core kernel serves it."""
    torch, la, orc = env
    h_max = max(h for h in range(1, 129) if la.la_prefill_path(1, h, 300) == 0)
    assert h_max >= 64, h_max
    assert all(la.la_prefill_path(1, h, 300) == -la.LA_ERR_UNSUPPORTED
               for h in range(h_max + 1, h_max + 4))
    _check_prefill(env, 1, 300, h_max, "bf16", 0.5, 17, simt=False)
    q, k, v, g = _inputs(torch, 1, 300, h_max + 1, torch.bfloat16, 0.5, 18)
    with pytest.raises(la.LaError) as e:
        la.la_prefill(q, k, v, g)
    assert e.value.status == la.LA_ERR_UNSUPPORTED
    _check_prefill(env, 1, 300, h_max + 1, "bf16", 0.5, 18, simt=True)


@pytest.mark.parametrize("H,N,S0", [(8, 40000, False), (4, 33000, True), (16, 50000, False)])
def test_segment_parallel_mode(env, H, N, S0):
    """One long sequence with few heads runs as segments side by side (the blockwise
    route's prefix over the d x d states), each from the state of the tokens before it;
    out, y and the final state against the oracle.  N has a ragged last chunk."""
    torch, la, _ = env
    assert la.la_prefill_path(1, H, N) == 2
    _check_prefill(env, 1, N, H, "bf16", 0.5, 700 + H, simt=False, S0=S0)


def test_segment_parallel_mode_repeatable_and_in_place(env):
    """The segment mode is deterministic, takes kv_state_out == kv_state_in, and agrees
    with the serial chain to the parity tolerance (only the order of fp32 state
    additions differs)."""
    torch, la, _ = env
    B, N, H = 1, 40000, 8
    q, k, v, g = _inputs(torch, B, N, H, torch.bfloat16, 0.5, 811)
    gen = torch.Generator(device="cuda").manual_seed(812)
    S_in = torch.randn((B, H, 128, 128), generator=gen, device="cuda") * 0.5
    out1, S1 = la.la_prefill(q, k, v, g, kv_state_in=S_in)
    out2, S2 = la.la_prefill(q, k, v, g, kv_state_in=S_in)
    S_io = S_in.clone()
    out3, _ = la.la_prefill(q, k, v, g, kv_state_in=S_io, kv_state_out=S_io)
    out_s, S_s = la.la_prefill(q, k, v, g, kv_state_in=S_in, serial=True)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    assert torch.equal(out1, out2) and torch.equal(S1, S2)
    assert torch.equal(out3, out1) and torch.equal(S_io, S1)
    assert rel_max_err(host64(out1), host64(out_s)) <= TOL["bf16"]["out"]
    assert rel_max_err(host64(S1), host64(S_s)) <= TOL["bf16"]["state"]


def test_prefill_8k_workload_full(env):
    """B1 H64 N8192 d128 bf16, inputs N(0,1)*0.5: every output and the final state."""
    from linear_attention_hybrid_fwd_b300.inputs import WORKLOADS
    w = WORKLOADS["prefill_8k"]
    _check_prefill(env, w.B, w.N, w.H, "bf16", w.scale, w.seed, simt=False, per_head=True)


def _check_long_windows(env, name, n_windows, slab=8192, want_y=False):
    """Long prefill: the whole sequence runs on the GPU; the oracle carries the fp64
    state through the sequence in slabs (oracle.state_pass, all heads) and runs the
    full layer on ``n_windows`` seeded 4096-token windows from the state at each
    window's start.  Each window is checked on all heads (the norm spans them) and on
    one seeded head; the final state on every head."""
    torch, la, orc = env
    from oracle.state_pass import state_pass
    from linear_attention_hybrid_fwd_b300.inputs import WORKLOADS
    w = WORKLOADS[name]
    q, k, v, g = _inputs(torch, w.B, w.N, w.H, torch.bfloat16, w.scale, w.seed)
    y = (torch.empty((w.B, w.N, w.H, 128), device="cuda", dtype=torch.float32)
         if want_y else None)
    out, S = la.la_prefill(q, k, v, g, y_debug=y)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    assert la.la_prefill_path(w.B, w.H, w.N) == 0
    rng = np.random.default_rng(w.seed)
    W = 4096
    starts = sorted(int(s) for s in rng.integers(0, w.N - W, size=n_windows))
    heads = [int(x) for x in rng.integers(0, w.H, size=n_windows)]
    S_run = np.zeros((w.B, w.H, 128, 128))
    pos = 0
    for t0, hsel in zip(starts + [w.N], heads + [None]):
        while pos < t0:  # state-only pass over [pos, t0)
            e = min(t0, pos + slab)
            S_run = state_pass(k[:, pos:e].cpu(), v[:, pos:e].cpu(), S_run)
            pos = e
        if hsel is None:
            break
        sl = slice(t0, t0 + W)
        ref_out, ref_y, _ = orc.prefill(host64(q[:, sl]), host64(k[:, sl]),
                                        host64(v[:, sl]), host64(g[:, sl]), S0=S_run)
        if want_y:  # pre-norm y of the window, per token row of H*d features
            e_y = row_rel_err(host64(y[:, sl]), ref_y, axes=(-2, -1))
            assert e_y <= TOL["bf16"]["y_row"], f"window {t0}: y token-row err {e_y:.3e}"

        got = host64(out[:, sl])
        e_all = rel_max_err(got, ref_out)
        e_head = rel_max_err(got[:, :, hsel], ref_out[:, :, hsel])
        assert e_all <= TOL["bf16"]["out"], f"window {t0}: out rel err {e_all:.3e}"
        assert e_head <= TOL["bf16"]["out"], f"window {t0} head {hsel}: {e_head:.3e}"
    e_S = rel_max_err(host64(S), S_run)
    assert e_S <= TOL["bf16"]["state"], f"final state rel err {e_S:.3e}"
    for h in range(w.H):
        assert rel_max_err(host64(S[:, h]), S_run[:, h]) <= TOL["bf16"]["state"], h


def test_prefill_128k_workload_windows(env):
    """B1 H64 N131072 d128 bf16: two seeded windows (output and pre-norm y) and the final
    state."""
    _check_long_windows(env, "prefill_128k", 2, want_y=True)


def test_prefill_1m_workload_windows(env):
    """B1 H64 N1048576 d128 bf16 (about 84 GB of I/O): eight seeded (head, 4096-token
    window) slices and the final per-head state."""
    torch, _, _ = env
    free, _ = torch.cuda.mem_get_info()
    assert free > 100 * 2**30, "the 1M-token workload needs about 90 GB of device memory"
    _check_long_windows(env, "prefill_1m", 8)


@pytest.mark.parametrize("simt", [False, True])
def test_split_prefill_continuation(env, simt):
    """Prefill of [0, N) equals prefill of [0, c) then [c, N) from the carried state."""
    torch, la, orc = env
    q, k, v, g = _inputs(torch, 1, 700, 4, torch.bfloat16, 0.5, 41)
    out, S = la.la_prefill(q, k, v, g, simt=simt)
    c = 333
    sl1, sl2 = slice(0, c), slice(c, 700)
    p = [t[:, sl1].contiguous() for t in (q, k, v, g)]
    o1, S1 = la.la_prefill(*p, simt=simt)
    p = [t[:, sl2].contiguous() for t in (q, k, v, g)]
    o2, S2 = la.la_prefill(*p, kv_state_in=S1, simt=simt)
    torch.cuda.synchronize()
    ref = host64(out)
    assert rel_max_err(np.concatenate([host64(o1), host64(o2)], 1), ref) <= 1e-2
    assert rel_max_err(host64(S2), host64(S)) <= 1e-5


@pytest.mark.parametrize("simt", [False, True])
def test_deterministic(env, simt):
    torch, la, _ = env
    q, k, v, g = _inputs(torch, 1, 600, 8, torch.bfloat16, 0.5, 51)
    o1, S1 = la.la_prefill(q, k, v, g, simt=simt)
    o2, S2 = la.la_prefill(q, k, v, g, simt=simt)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_n0_copies_or_zeroes_state(env):
    torch, la, _ = env
    q = torch.empty((1, 0, 2, 128), device="cuda", dtype=torch.bfloat16)
    S_in = torch.randn((1, 2, 128, 128), device="cuda")
    out, S = la.la_prefill(q, q, q, q, kv_state_in=S_in)
    torch.cuda.synchronize()
    assert torch.equal(S, S_in)
    _, S0 = la.la_prefill(q, q, q, q)
    torch.cuda.synchronize()
    assert torch.count_nonzero(S0) == 0


@pytest.mark.parametrize("simt", [False, True])
def test_guard_bands_untouched(env, simt):
    """Outputs written into the middle of larger buffers leave the sentinels intact."""
    torch, la, _ = env
    B, N, H, d = 1, 300, 4, 128
    q, k, v, g = _inputs(torch, B, N, H, torch.bfloat16, 0.5, 61)
    n = B * N * H * d
    pad = 4096
    ob = torch.full((n + 2 * pad,), 7.0, device="cuda", dtype=torch.bfloat16)
    sb = torch.full((B * H * d * d + 2 * pad,), -3.0, device="cuda", dtype=torch.float32)
    out = ob[pad:pad + n].view(B, N, H, d)
    S = sb[pad:pad + B * H * d * d].view(B, H, d, d)
    la.la_prefill(q, k, v, g, out=out, kv_state_out=S, simt=simt)
    torch.cuda.synchronize()
    assert torch.all(ob[:pad] == 7.0) and torch.all(ob[pad + n:] == 7.0)
    assert torch.all(sb[:pad] == -3.0) and torch.all(sb[-pad:] == -3.0)
