"""Pins for the fp64 input-projection oracle (oracle/projection.py).

The projection ("Hybrid Modeling", MiniMax-01 deep dive: step 1 "Input X", step 2
"Q, K, V = SiLU(X)", read as q, k, v, g = x W_{q,k,v,g}^T with SiLU on q, k, v) is
checked against things other than itself:

* pure-Python triple loops on tiny shapes (no library matrix product)
* the segment order of the stacked weight and where SiLU applies, with constant rows
  whose outputs have closed forms; SiLU's value there from the tanh form
  x/2 (1 + tanh(x/2)), a different route from x / (1 + e^-x)
* identity weights give the input's own features back
* linearity in x and in W (raw outputs)
* the activated outputs fed to the layer's core equal the raw outputs fed to the
  layer (SiLU is applied once, in one place)
A transposed weight, swapped segments, SiLU on g, or a wrong head reshape fails one.
"""
import math

import numpy as np
import pytest

from oracle.projection import project, silu


def _loops(x, w, H, d):
    T, hidden = len(x), len(x[0])
    HD = H * d
    outs = []
    for s in range(4):
        o = np.zeros((T, H, d))
        for t in range(T):
            for h in range(H):
                for j in range(d):
                    acc = 0.0
                    for i in range(hidden):
                        acc += x[t][i] * w[s * HD + h * d + j][i]
                    o[t, h, j] = acc
        outs.append(o)
    return outs


@pytest.mark.parametrize("T,hidden,H,d", [(1, 1, 1, 1), (3, 5, 1, 2), (4, 7, 2, 3)])
def test_projection_matches_loops(T, hidden, H, d):
    rng = np.random.default_rng(T * 100 + hidden)
    x = rng.standard_normal((T, hidden))
    w = rng.standard_normal((4 * H * d, hidden))
    got = project(x, w, H, d, activate=False)
    want = _loops(x.tolist(), w.tolist(), H, d)
    for s in range(4):
        np.testing.assert_allclose(got[s], want[s], rtol=1e-13, atol=1e-13)


def _silu_tanh(c):
    return 0.5 * c * (1.0 + math.tanh(0.5 * c))


def test_segment_order_and_activation_placement():
    # x = ones; every row of segment s is (s + 1) / 4 and hidden = 4, so the raw
    # outputs are exactly 1, 2, 3, 4 for q, k, v, g (quarters are exact in binary).
    H, d, hidden, T = 2, 2, 4, 3
    x = np.ones((T, hidden))
    w = np.concatenate([np.full((H * d, hidden), (s + 1) / hidden) for s in range(4)])
    q, k, v, g = project(x, w, H, d, activate=False)
    for o, c in zip((q, k, v, g), (1.0, 2.0, 3.0, 4.0)):
        assert np.array_equal(o, np.full((T, H, d), c))
    q, k, v, g = project(x, w, H, d, activate=True)
    for o, c in zip((q, k, v), (1.0, 2.0, 3.0)):
        np.testing.assert_allclose(o, _silu_tanh(c), rtol=1e-15)
    assert np.array_equal(g, np.full((T, H, d), 4.0)), "g must stay raw"


def test_head_reshape_is_feature_major():
    # feature f = h*d + j of a segment comes from weight row s*H*d + f
    H, d, hidden = 3, 4, 12
    x = np.eye(hidden)[:1]                      # picks column 0 of every weight row
    w = np.zeros((4 * H * d, hidden))
    w[:, 0] = np.arange(4 * H * d)
    q, k, v, g = project(x, w, H, d, activate=False)
    for s, o in enumerate((q, k, v, g)):
        for h in range(H):
            for j in range(d):
                assert o[0, h, j] == s * H * d + h * d + j


def test_identity_weights_return_features():
    rng = np.random.default_rng(3)
    H, d, T = 2, 4, 5
    hidden = 3 * H * d
    x = rng.standard_normal((T, hidden))
    w = np.zeros((4 * H * d, hidden))
    HD = H * d
    w[0:HD, 0:HD] = np.eye(HD)                  # q = x[:, 0:HD]
    w[HD:2 * HD, HD:2 * HD] = np.eye(HD)        # k = x[:, HD:2HD]
    w[2 * HD:3 * HD, 2 * HD:3 * HD] = np.eye(HD)
    w[3 * HD:4 * HD, 0:HD] = -np.eye(HD)        # g = -x[:, 0:HD]
    q, k, v, g = project(x, w, H, d, activate=False)
    assert np.array_equal(q.reshape(T, HD), x[:, :HD])
    assert np.array_equal(k.reshape(T, HD), x[:, HD:2 * HD])
    assert np.array_equal(v.reshape(T, HD), x[:, 2 * HD:])
    assert np.array_equal(g.reshape(T, HD), -x[:, :HD])


def test_linearity_in_x_and_w():
    rng = np.random.default_rng(4)
    H, d, hidden, T = 2, 3, 5, 4
    x1, x2 = rng.standard_normal((2, T, hidden))
    w1, w2 = rng.standard_normal((2, 4 * H * d, hidden))
    a, b = 0.75, -1.5
    lhs = project(a * x1 + b * x2, w1, H, d, activate=False)
    r1 = project(x1, w1, H, d, activate=False)
    r2 = project(x2, w1, H, d, activate=False)
    for s in range(4):
        np.testing.assert_allclose(lhs[s], a * r1[s] + b * r2[s], rtol=1e-12, atol=1e-12)
    lhs = project(x1, a * w1 + b * w2, H, d, activate=False)
    r2 = project(x1, w2, H, d, activate=False)
    for s in range(4):
        np.testing.assert_allclose(lhs[s], a * r1[s] + b * r2[s], rtol=1e-12, atol=1e-12)


def test_activated_outputs_feed_the_core(oracle_mod):
    """The layer on raw projections (SiLU inside the layer) equals the core + norm/gate
    on the activated projections: SiLU happens exactly once."""
    rng = np.random.default_rng(5)
    H, d, hidden, T = 2, 4, 6, 9
    x = rng.standard_normal((T, hidden))
    w = rng.standard_normal((4 * H * d, hidden)) * 0.5
    raw = [o[None] for o in project(x, w, H, d, activate=False)]
    act = [o[None] for o in project(x, w, H, d, activate=True)]
    out_raw, _, S_raw = oracle_mod.prefill(*raw)
    y, S_act = oracle_mod.core(*act[:3])
    out_act = oracle_mod.rmsnorm_gate(y, act[3])
    np.testing.assert_allclose(out_raw, out_act, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_raw, S_act, rtol=1e-12, atol=1e-12)


def test_silu_extremes():
    assert silu(0.0) == 0.0
    assert silu(-800.0) == 0.0                  # e^800 overflows: -800 / inf
    assert silu(40.0) == 40.0                   # 1 + e^-40 rounds to 1
