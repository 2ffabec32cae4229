"""Pins for the fp64 softmax-attention oracle (oracle/softmax_attn.py).

The layer: RoPE on the first half of each head's features (base 1e7, "rotate half"
pairs), then causal softmax(q k^T / sqrt(d)) v.  Checked against things other than
the code itself:

* RoPE: identity at position 0; a hand-worked rotation; each rotated pair keeps its
  norm and the other half passes unchanged; the dot product of a rotated query and key
  depends only on their distance (the property RoPE exists for)
* attention: pure-Python loops on tiny shapes; the first token attends only to itself
  (o_0 = v_0); q = 0 gives the running mean of v; very large scores pick the
  best-matching key (no overflow)
A wrong pairing, a sign slip in the rotation, exclusive causality, a missing 1/sqrt(d)
or a transposed score matrix fails one of them.
"""
import math

import numpy as np
import pytest

from oracle.softmax_attn import attention, rope


def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 1, 3, 16))
    assert np.array_equal(rope(x), x)


def test_rope_hand_worked():
    # d = 8: pairs (0, 2) with theta_0 = 1 and (1, 3) with theta_1 = base^(-1/2) = 0.1
    x = np.zeros((1, 3, 1, 8))
    x[0, 2, 0] = [1.0, 2.0, 0.0, 0.0, 5.0, 6.0, 7.0, 8.0]
    r = rope(x, base=100.0)[0, 2, 0]
    # token 2: pair 0 rotated by 2 rad, pair 1 by 0.2 rad
    np.testing.assert_allclose(r[[0, 2]], [math.cos(2.0), math.sin(2.0)], rtol=1e-15)
    np.testing.assert_allclose(r[[1, 3]], [2 * math.cos(0.2), 2 * math.sin(0.2)], rtol=1e-15)
    assert np.array_equal(r[4:], [5.0, 6.0, 7.0, 8.0])


def test_rope_keeps_pair_norms_and_second_half():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((1, 50, 2, 128))
    r = rope(x)
    np.testing.assert_allclose(r[..., :32] ** 2 + r[..., 32:64] ** 2,
                               x[..., :32] ** 2 + x[..., 32:64] ** 2, rtol=1e-12)
    assert np.array_equal(r[..., 64:], x[..., 64:])


def test_rope_relative_position():
    rng = np.random.default_rng(3)
    d, N = 16, 12
    qv, kv = rng.standard_normal((2, d))
    q = np.broadcast_to(qv, (1, N, 1, d)).copy()
    k = np.broadcast_to(kv, (1, N, 1, d)).copy()
    D = rope(q, base=50.0)[0, :, 0] @ rope(k, base=50.0)[0, :, 0].T
    for t1 in range(N - 1):
        for t2 in range(N - 1):
            assert abs(D[t1 + 1, t2 + 1] - D[t1, t2]) < 1e-12
    assert abs(D[3, 1] - D[1, 3]) > 1e-3        # but not on the sign of the distance


def _loops(q, k, v, base):
    qr, kr = rope(q, base), rope(k, base)
    B, N, H, d = q.shape
    out = np.zeros((B, N, H, d))
    for b in range(B):
        for h in range(H):
            for t in range(N):
                sc = [sum(qr[b, t, h, i] * kr[b, s, h, i] for i in range(d)) / math.sqrt(d)
                      for s in range(t + 1)]
                m = max(sc)
                w = [math.exp(x - m) for x in sc]
                z = sum(w)
                for j in range(d):
                    out[b, t, h, j] = sum(w[s] * v[b, s, h, j] for s in range(t + 1)) / z
    return out


@pytest.mark.parametrize("B,N,H,d", [(1, 1, 1, 4), (1, 5, 2, 8), (2, 7, 1, 12)])
def test_attention_matches_loops(B, N, H, d):
    rng = np.random.default_rng(B * 100 + N)
    q, k, v = rng.standard_normal((3, B, N, H, d))
    np.testing.assert_allclose(attention(q, k, v, base=30.0), _loops(q, k, v, 30.0),
                               rtol=1e-12, atol=1e-12)


def test_first_token_attends_to_itself():
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((3, 2, 9, 3, 16))
    o = attention(q, k, v)
    assert np.array_equal(o[:, 0], v[:, 0])


def test_zero_query_gives_running_mean():
    rng = np.random.default_rng(5)
    k, v = rng.standard_normal((2, 1, 20, 2, 8))
    o = attention(np.zeros_like(k), k, v)
    want = np.cumsum(v, axis=1) / np.arange(1, 21)[None, :, None, None]
    np.testing.assert_allclose(o, want, rtol=1e-13, atol=1e-14)


def test_large_scores_select_the_best_key():
    # keys are +-e_j scaled by 1e3 at the unrotated features; the query matches key 2
    d = 8
    k = np.zeros((1, 4, 1, d))
    for s in range(4):
        k[0, s, 0, 4 + s] = 1e3
    q = np.zeros((1, 4, 1, d))
    q[0, 3, 0, 6] = 1e3                          # token 3 matches key 2 with score 5e5
    v = np.arange(4 * d, dtype=np.float64).reshape(1, 4, 1, d)
    o = attention(q, k, v)
    assert np.all(np.isfinite(o))
    assert np.array_equal(o[0, 3, 0], v[0, 2, 0])
