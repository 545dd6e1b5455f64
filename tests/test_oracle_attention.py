"""Pins of the fp64 attention: closed forms, the softmax's shift invariance,
causal special cases, and agreement with an independent per-element loop."""
import math

import numpy as np

from oracle import attention as A


def _loop_attention(Q, K, V, scale, causal):
    # the definition element by element: O[i][c] = sum_j e^{s_ij - m_i} V[j][c] / sum_j e^{s_ij - m_i}
    Sq, d = Q.shape
    Sk = K.shape[0]
    O = np.zeros((Sq, V.shape[1]))
    for i in range(Sq):
        keys = [j for j in range(Sk) if not causal or j <= i + (Sk - Sq)]
        if not keys:
            continue
        s = {j: scale * sum(Q[i, t] * K[j, t] for t in range(d)) for j in keys}
        m = max(s.values())
        w = {j: math.exp(s[j] - m) for j in keys}
        den = sum(w.values())
        for c in range(V.shape[1]):
            O[i, c] = sum(w[j] * V[j, c] for j in keys) / den
    return O


def test_matches_loop_definition():
    rng = np.random.default_rng(1)
    for causal, (Sq, Sk) in ((False, (5, 7)), (True, (6, 6)), (True, (3, 8))):
        Q = rng.standard_normal((1, 2, Sq, 4))
        K = rng.standard_normal((1, 1, Sk, 4))    # grouped: both query heads read head 0
        V = rng.standard_normal((1, 1, Sk, 3))
        O = A.attention(Q, K, V, 0.7, causal)
        for h in range(2):
            want = _loop_attention(Q[0, h], K[0, 0], V[0, 0], 0.7, causal)
            assert np.allclose(O[0, h], want, rtol=1e-13, atol=1e-14)


def test_equal_keys_average_the_values():
    # identical keys: every score in a row is equal, P is uniform, O is the mean of V
    rng = np.random.default_rng(2)
    Q = rng.standard_normal((1, 1, 4, 8))
    K = np.tile(rng.standard_normal((1, 1, 1, 8)), (1, 1, 6, 1))
    V = rng.standard_normal((1, 1, 6, 5))
    O = A.attention(Q, K, V)
    assert np.allclose(O[0, 0], np.tile(V[0, 0].mean(axis=0), (4, 1)), rtol=1e-14, atol=1e-15)


def test_dominant_key_selects_its_value():
    Q = np.zeros((1, 1, 1, 2)); Q[..., 0] = 1.0
    K = np.zeros((1, 1, 3, 2)); K[0, 0, 1, 0] = 100.0          # s = (0, 100/sqrt2, 0) * ...
    V = np.arange(9.0).reshape(1, 1, 3, 3)
    O = A.attention(Q, K, V, scale=1.0)
    assert np.allclose(O[0, 0, 0], V[0, 0, 1], rtol=0, atol=1e-40)


def test_shift_invariance_of_the_softmax():
    # appending a component c to q and 1 to every k adds c to every score of a
    # row: the output must not change
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((1, 1, 5, 4)); K = rng.standard_normal((1, 1, 7, 4))
    V = rng.standard_normal((1, 1, 7, 4))
    Q2 = np.concatenate([Q, np.full((1, 1, 5, 1), 3.0)], axis=3)
    K2 = np.concatenate([K, np.ones((1, 1, 7, 1))], axis=3)
    assert np.allclose(A.attention(Q, K, V, 0.5), A.attention(Q2, K2, V, 0.5), rtol=1e-12, atol=1e-13)


def test_causal_first_row_and_default_scale():
    rng = np.random.default_rng(4)
    Q = rng.standard_normal((1, 1, 4, 16)); K = rng.standard_normal((1, 1, 4, 16))
    V = rng.standard_normal((1, 1, 4, 6))
    O = A.attention(Q, K, V, causal=True)
    assert np.allclose(O[0, 0, 0], V[0, 0, 0], rtol=0, atol=0)   # only key 0 is visible
    assert np.allclose(A.attention(Q, K, V), A.attention(Q, K, V, 0.25))   # 1/sqrt(16)
    # more queries than keys under the causal alignment: early rows see nothing
    O = A.attention(rng.standard_normal((1, 1, 5, 2)), K[..., :2], V, causal=True)
    assert not O[0, 0, 0].any()


def test_error_scale_bounds_the_output():
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((2, 2, 6, 8)); K = rng.standard_normal((2, 2, 9, 8))
    V = rng.standard_normal((2, 2, 9, 8))
    s = A.error_scale(Q, K, V, causal=True)
    assert np.abs(A.attention(Q, K, V, causal=True)).max() <= s <= np.abs(V).max()
