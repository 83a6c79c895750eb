"""Pins for oracle.layernorm: closed forms, invariances, brute-force loops."""
import numpy as np

from oracle.layernorm import layernorm

rng = np.random.default_rng(11)


def test_closed_forms():
    # row [-1, 1]: mean 0, variance 1 -> y = x * gamma + beta (eps = 0)
    y, mu, rs = layernorm(np.array([[-1.0, 1.0]]), [2.0, 3.0], [0.5, -0.5], 0.0)
    np.testing.assert_array_equal(mu, [0.0])
    np.testing.assert_array_equal(rs, [1.0])
    np.testing.assert_array_equal(y, [[-1.5, 2.5]])
    # a constant row normalises to beta; its rsigma is 1 / sqrt(eps)
    y, mu, rs = layernorm(np.full((1, 8), 7.0), np.ones(8), np.arange(8.0), 1e-4)
    np.testing.assert_array_equal(y, [np.arange(8.0)])
    np.testing.assert_allclose(rs, [100.0], rtol=1e-15)


def test_shift_and_scale_invariance():
    x = rng.standard_normal((5, 64))
    g, b = rng.standard_normal(64), rng.standard_normal(64)
    y0, _, _ = layernorm(x, g, b, 0.0)
    y1, _, _ = layernorm(3.5 * x - 2.0, g, b, 0.0)
    np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=1e-12)
    # unit gamma, zero beta: every row has mean 0 and variance 1
    y, _, _ = layernorm(x, np.ones(64), np.zeros(64), 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, rtol=1e-12)


def test_brute_force_loops():
    x = rng.standard_normal((3, 6))
    g, b, eps = rng.standard_normal(6), rng.standard_normal(6), 1e-5
    y, mu, rs = layernorm(x, g, b, eps)
    for r in range(3):
        m = sum(x[r]) / 6
        v = sum((t - m) ** 2 for t in x[r]) / 6
        s = 1.0 / (v + eps) ** 0.5
        assert abs(mu[r] - m) < 1e-14 and abs(rs[r] - s) < 1e-12 * s
        for c in range(6):
            assert abs(y[r, c] - ((x[r, c] - m) * s * g[c] + b[c])) < 1e-12
