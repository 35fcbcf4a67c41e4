"""Pins of the oracle's packed linear layer (CPU only): brute-force sums,
an identity weight, linearity, and the rows it covers."""
from __future__ import annotations

import numpy as np

import oracle


def test_brute_force_sums():
    rng = np.random.default_rng(7)
    cap, K, N, T = 7, 5, 3, 4
    a = rng.standard_normal((cap, K))
    w = rng.standard_normal((N, K))
    bias = rng.standard_normal(N)
    out = oracle.linear_packed(a, w, bias, T)
    assert out.shape == (T, N)
    for t in range(T):
        for n in range(N):
            s = bias[n]
            for k in range(K):
                s += a[t, k] * w[n, k]
            assert abs(out[t, n] - s) < 1e-12


def test_identity_weight_copies_rows_and_no_bias():
    rng = np.random.default_rng(8)
    a = rng.standard_normal((9, 6))
    out = oracle.linear_packed(a, np.eye(6), None, 9)
    assert np.array_equal(out, a)
    assert oracle.linear_packed(a, np.eye(6), None, 0).shape == (0, 6)


def test_linearity_in_rows_and_weights():
    rng = np.random.default_rng(9)
    a1, a2 = rng.standard_normal((2, 5, 8))
    w1, w2 = rng.standard_normal((2, 4, 8))
    f = lambda a, w: oracle.linear_packed(a, w, None, 5)
    assert np.allclose(f(a1 + 2 * a2, w1), f(a1, w1) + 2 * f(a2, w1))
    assert np.allclose(f(a1, w1 - w2), f(a1, w1) - f(a1, w2))
