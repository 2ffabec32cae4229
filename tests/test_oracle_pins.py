"""Pins for the fp64 oracle: each checks it against something other than itself.

The method (MiniMax-01 deep dive, Hugging Face blog, "Hybrid Modeling", mechanism
steps 2-4): q^,k^,v^ = SiLU(q,k,v); Y = Q^ (K^T V) taken causally through the d x d
state; out = RMSNorm(Y) * sigmoid(G).  Pins used here:

* a hand-worked recurrence and a hand-worked norm/gate example (``tests/golden``)
* the quadratic masked form (Q^ K^T * M) V^ by brute force (a different algorithm)
* closed forms: first token, constant inputs, d = 1 prefix sums
* the final state equals an independent K^T V product
* invariants: linearity, split prefill == whole prefill, prefill state == N decode
  steps, head permutation equivariance, eps = 0 scale invariance, g -> +inf
* SiLU against the tanh form x/2 (1 + tanh(x/2)) and its odd-part identity
Each pin is chosen so that a plausible slip (a dropped term, exclusive instead of
inclusive causality, a transposed state, a wrong norm width, SiLU on g) fails it.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(x) for x in rest])
    return vals


def _rand(rng, shape, scale=1.0):
    return rng.standard_normal(shape) * scale


# ----------------------------------------------------------------------------- SiLU
def test_silu_against_tanh_form(oracle_mod):
    x = np.linspace(-30, 30, 2001)
    ref = 0.5 * x * (1.0 + np.tanh(0.5 * x))  # same function, different formula
    # (1 + tanh) cancels for x << 0, so the tanh form is only good to ~1e-15 absolute
    np.testing.assert_allclose(oracle_mod.silu(x), ref, rtol=1e-13, atol=1e-14)
    xn = np.linspace(-30, -5, 101)  # the negative tail: x e^x / (1 + e^x)
    np.testing.assert_allclose(oracle_mod.silu(xn), xn * np.exp(xn) / (1 + np.exp(xn)),
                               rtol=1e-13)


def test_silu_identities(oracle_mod):
    x = np.linspace(-20, 20, 401)
    s = oracle_mod.silu(x)
    sn = oracle_mod.silu(-x)
    np.testing.assert_allclose(s - sn, x, atol=1e-12)  # x(sigma(x) + sigma(-x)) = x
    assert oracle_mod.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(oracle_mod.silu(np.array([50.0])), [50.0], rtol=1e-15)
    assert np.all(s >= -0.2785)  # global minimum of SiLU is about -0.27846


# ------------------------------------------------------------------ worked examples
def test_core_worked_example(oracle_mod):
    fx = _read_fixture("core_worked_example.txt")
    N, d = int(fx["N"][0]), int(fx["d"][0])
    q, k, v = (fx[n].reshape(1, N, 1, d) for n in "qkv")
    y, S = oracle_mod.core(q, k, v)
    np.testing.assert_array_equal(y.reshape(N, d), fx["y"].reshape(N, d))
    np.testing.assert_array_equal(S.reshape(d, d), fx["S"].reshape(d, d))


def test_norm_gate_worked_example(oracle_mod):
    fx = _read_fixture("norm_gate_worked_example.txt")
    y = fx["y"].reshape(1, 1, 1, 2)
    g = fx["g"].reshape(1, 1, 1, 2)
    out = oracle_mod.rmsnorm_gate(y, g, eps=float(fx["eps"][0]))
    np.testing.assert_allclose(out.ravel(), fx["out"], rtol=1e-14)


# ---------------------------------------------------------------- quadratic form
def _quadratic(qh, kh, vh):
    """Brute force Y = (Q^ K^T * M) V^ with M[t,s] = 1 iff s <= t, per (b,h)."""
    B, N, H, d = qh.shape
    y = np.zeros_like(qh)
    M = np.tril(np.ones((N, N)))
    for b in range(B):
        for h in range(H):
            A = qh[b, :, h, :] @ kh[b, :, h, :].T
            y[b, :, h, :] = (A * M) @ vh[b, :, h, :]
    return y


@pytest.mark.parametrize("B,N,H,d", [(1, 1, 1, 1), (1, 17, 1, 1), (2, 33, 3, 2), (1, 64, 2, 4),
                                     (1, 40, 1, 8), (2, 9, 2, 16), (1, 48, 1, 128)])
def test_core_matches_quadratic(oracle_mod, B, N, H, d):
    rng = np.random.default_rng(100 + N * 7 + d)
    qh, kh, vh = (_rand(rng, (B, N, H, d)) for _ in range(3))
    y, S = oracle_mod.core(qh, kh, vh)
    ref = _quadratic(qh, kh, vh)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())


def test_prefill_matches_quadratic_pipeline(oracle_mod):
    """Whole layer: tanh-form SiLU -> quadratic form -> numpy RMSNorm * sigmoid."""
    rng = np.random.default_rng(7)
    B, N, H, d = 2, 24, 3, 8
    q, k, v, g = (_rand(rng, (B, N, H, d)) for _ in range(4))
    act = lambda x: 0.5 * x * (1.0 + np.tanh(0.5 * x))
    y = _quadratic(act(q), act(k), act(v))
    ms = (y.reshape(B, N, H * d) ** 2).mean(-1)
    ref = y / np.sqrt(ms + 1e-6)[:, :, None, None] * (0.5 * (1.0 + np.tanh(0.5 * g)))
    out, ypre, S = oracle_mod.prefill(q, k, v, g, eps=1e-6)
    np.testing.assert_allclose(ypre, y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- closed forms
def test_first_token_closed_form(oracle_mod):
    rng = np.random.default_rng(1)
    qh, kh, vh = (_rand(rng, (1, 5, 2, 16)) for _ in range(3))
    y, _ = oracle_mod.core(qh, kh, vh)
    for h in range(2):
        want = np.dot(qh[0, 0, h], kh[0, 0, h]) * vh[0, 0, h]
        np.testing.assert_allclose(y[0, 0, h], want, rtol=1e-13)


def test_constant_inputs_closed_form(oracle_mod):
    rng = np.random.default_rng(2)
    d, N = 8, 300
    a, b, c = rng.standard_normal(d), rng.standard_normal(d), rng.standard_normal(d)
    qh = np.broadcast_to(a, (1, N, 1, d))
    kh = np.broadcast_to(b, (1, N, 1, d))
    vh = np.broadcast_to(c, (1, N, 1, d))
    y, S = oracle_mod.core(qh, kh, vh)
    t1 = np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(y[0, :, 0, :], t1 * np.dot(a, b) * c[None, :], rtol=1e-11)
    np.testing.assert_allclose(S[0, 0], N * np.outer(b, c), rtol=1e-12)


def test_d1_is_prefix_sum(oracle_mod):
    rng = np.random.default_rng(3)
    N = 257
    qh, kh, vh = (_rand(rng, (1, N, 1, 1)) for _ in range(3))
    y, S = oracle_mod.core(qh, kh, vh)
    want = qh.ravel() * np.cumsum(kh.ravel() * vh.ravel())
    np.testing.assert_allclose(y.ravel(), want, rtol=1e-12, atol=1e-12)


def test_final_state_is_KtV(oracle_mod):
    rng = np.random.default_rng(4)
    B, N, H, d = 2, 37, 3, 16
    qh, kh, vh = (_rand(rng, (B, N, H, d)) for _ in range(3))
    S0 = _rand(rng, (B, H, d, d))
    _, S = oracle_mod.core(qh, kh, vh, S0=S0)
    for b in range(B):
        for h in range(H):
            want = S0[b, h] + kh[b, :, h, :].T @ vh[b, :, h, :]
            np.testing.assert_allclose(S[b, h], want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariants
def test_linearity_in_v_and_q(oracle_mod):
    rng = np.random.default_rng(5)
    shp = (1, 20, 2, 8)
    qh, kh, v1, v2, q2 = (_rand(rng, shp) for _ in range(5))
    a, b = 1.7, -0.3
    y1, _ = oracle_mod.core(qh, kh, v1)
    y2, _ = oracle_mod.core(qh, kh, v2)
    y12, _ = oracle_mod.core(qh, kh, a * v1 + b * v2)
    np.testing.assert_allclose(y12, a * y1 + b * y2, rtol=1e-11, atol=1e-11)
    yq2, _ = oracle_mod.core(q2, kh, v1)
    yq12, _ = oracle_mod.core(a * qh + b * q2, kh, v1)
    np.testing.assert_allclose(yq12, a * y1 + b * yq2, rtol=1e-11, atol=1e-11)


def test_split_prefill_equals_whole(oracle_mod):
    rng = np.random.default_rng(6)
    B, N, H, d = 1, 50, 2, 8
    q, k, v, g = (_rand(rng, (B, N, H, d)) for _ in range(4))
    out, y, S = oracle_mod.prefill(q, k, v, g)
    cut = 23
    o1, y1, S1 = oracle_mod.prefill(q[:, :cut], k[:, :cut], v[:, :cut], g[:, :cut])
    o2, y2, S2 = oracle_mod.prefill(q[:, cut:], k[:, cut:], v[:, cut:], g[:, cut:], S0=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, S, rtol=1e-12)


def test_prefill_state_equals_decode_steps(oracle_mod):
    rng = np.random.default_rng(8)
    B, N, H, d = 2, 12, 3, 4
    q, k, v, g = (_rand(rng, (B, N, H, d)) for _ in range(4))
    out, y, S = oracle_mod.prefill(q, k, v, g)
    St = np.zeros((B, H, d, d))
    for t in range(N):
        o, yt, St = oracle_mod.decode_step(St, q[:, t], k[:, t], v[:, t], g[:, t])
        np.testing.assert_allclose(o, out[:, t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(St, S, rtol=1e-12)


def test_head_permutation_equivariance(oracle_mod):
    rng = np.random.default_rng(9)
    B, N, H, d = 1, 10, 4, 4
    q, k, v, g = (_rand(rng, (B, N, H, d)) for _ in range(4))
    perm = np.array([2, 0, 3, 1])
    out, _, S = oracle_mod.prefill(q, k, v, g)
    outp, _, Sp = oracle_mod.prefill(q[:, :, perm], k[:, :, perm], v[:, :, perm], g[:, :, perm])
    np.testing.assert_allclose(outp, out[:, :, perm], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(Sp, S[:, perm], rtol=1e-13)


def test_norm_spans_all_heads(oracle_mod):
    """Scaling one head's pre-norm output changes every head's normalised output."""
    rng = np.random.default_rng(10)
    y = _rand(rng, (1, 3, 4, 8))
    g = np.full_like(y, 30.0)
    o1 = oracle_mod.rmsnorm_gate(y, g, eps=0.0)
    y2 = y.copy()
    y2[:, :, 0] *= 3.0
    o2 = oracle_mod.rmsnorm_gate(y2, g, eps=0.0)
    assert np.all(np.abs(o2[:, :, 1:] - o1[:, :, 1:]) > 0)
    # closed form: with g -> +inf the gate is 1 and each token has unit mean square
    ms = (o1.reshape(3, 32) ** 2).mean(-1)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-12)


def test_norm_eps_closed_form(oracle_mod):
    rng = np.random.default_rng(11)
    y = _rand(rng, (2, 5, 3, 8), 0.01)
    g = _rand(rng, (2, 5, 3, 8))
    eps = 1e-4
    out = oracle_mod.rmsnorm_gate(y, g, eps=eps)
    sig = 0.5 * (1 + np.tanh(0.5 * g))
    ms = (y.reshape(10, 24) ** 2).mean(-1)
    got = ((out / sig).reshape(10, 24) ** 2).mean(-1)
    np.testing.assert_allclose(got, ms / (ms + eps), rtol=1e-12)


def test_scale_invariance_eps0(oracle_mod):
    """With eps = 0 the output does not change when v^ is scaled by a > 0."""
    rng = np.random.default_rng(12)
    qh, kh, vh, g = (_rand(rng, (1, 16, 2, 8)) for _ in range(4))
    y1, _ = oracle_mod.core(qh, kh, vh)
    y2, _ = oracle_mod.core(qh, kh, 5.0 * vh)
    o1 = oracle_mod.rmsnorm_gate(y1, g, eps=0.0)
    o2 = oracle_mod.rmsnorm_gate(y2, g, eps=0.0)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)


def test_gate_not_activated(oracle_mod):
    """g enters only through sigmoid(g): out / sigmoid(g) does not depend on g."""
    rng = np.random.default_rng(13)
    q, k, v, g1, g2 = (_rand(rng, (1, 6, 2, 4)) for _ in range(5))
    o1, _, _ = oracle_mod.prefill(q, k, v, g1)
    o2, _, _ = oracle_mod.prefill(q, k, v, g2)
    s = lambda g: 0.5 * (1 + np.tanh(0.5 * g))
    np.testing.assert_allclose(o1 / s(g1), o2 / s(g2), rtol=1e-12)


def test_threads_do_not_change_result(oracle_mod):
    rng = np.random.default_rng(14)
    qh, kh, vh = (_rand(rng, (2, 30, 5, 8)) for _ in range(3))
    y1, S1 = oracle_mod.core(qh, kh, vh, nthreads=1)
    y4, S4 = oracle_mod.core(qh, kh, vh, nthreads=4)
    np.testing.assert_array_equal(y1, y4)
    np.testing.assert_array_equal(S1, S4)


# ------------------------------------------------------- long-sequence state pass
def test_state_pass_matches_recurrence(oracle_mod):
    """The batched-matmul state pass ends where the C token recurrence ends."""
    from oracle.state_pass import state_pass
    rng = np.random.default_rng(15)
    B, N, H, d = 2, 77, 3, 16
    q, k, v, g = (_rand(rng, (B, N, H, d)) for _ in range(4))
    S0 = _rand(rng, (B, H, d, d))
    _, _, S_rec = oracle_mod.prefill(q, k, v, g, S0=S0)
    np.testing.assert_allclose(state_pass(k, v, S0), S_rec, rtol=1e-12, atol=1e-12)
    # chained over slabs, as the long-sequence tests use it
    S_run = None
    for a in range(0, N, 20):
        S_run = state_pass(k[:, a:a + 20], v[:, a:a + 20], S_run)
    _, _, S_zero = oracle_mod.prefill(q, k, v, g)
    np.testing.assert_allclose(S_run, S_zero, rtol=1e-12, atol=1e-12)


def test_state_pass_silu_is_textbook():
    from oracle.state_pass import silu64
    x = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(silu64(x).numpy(), 0.5 * x * (1 + np.tanh(0.5 * x)),
                               rtol=1e-13, atol=1e-14)
