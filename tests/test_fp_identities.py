"""Floating-point identities the kernels rely on (CPU).

The rotated amax folds the last Hadamard butterfly into the maximum:
max(|fl(a + b)|, |fl(a - b)|) == fl(|a| + |b|) for finite fp32 a, b (one of the two
exact sums is +-(|a| + |b|), the other is no larger in magnitude, and round-to-nearest-even
is symmetric and monotone).  Checked here on random pairs over a wide exponent range and
on ties, signed zeros, subnormals and near-overflow values.
"""
import numpy as np

f32 = np.float32


def _check(a, b):
    a = np.asarray(a, f32)
    b = np.asarray(b, f32)
    with np.errstate(over="ignore"):
        lhs = np.maximum(np.abs((a + b).astype(f32)), np.abs((a - b).astype(f32)))
        rhs = (np.abs(a) + np.abs(b)).astype(f32)
    assert np.array_equal(lhs.view(np.uint32), rhs.view(np.uint32))


def test_butterfly_abs_max_identity_random():
    rng = np.random.default_rng(7)
    n = 1 << 20
    mant = rng.standard_normal(n).astype(f32)
    a = (mant * np.exp2(rng.integers(-40, 40, n)).astype(f32)).astype(f32)
    b = (rng.standard_normal(n).astype(f32) * np.exp2(rng.integers(-40, 40, n)).astype(f32)).astype(f32)
    _check(a, b)
    # bf16-valued inputs (what the transform sees) at close exponents: many exact ties
    a16 = (a.view(np.uint32) & 0xFFFF0000).view(f32)
    b16 = (b.view(np.uint32) & 0xFFFF0000).view(f32)
    _check(a16, b16)


def test_butterfly_abs_max_identity_edges():
    tiny = np.finfo(f32).tiny
    mx = np.finfo(f32).max
    vals = np.array([0.0, -0.0, 1.0, -1.0, 1.5, tiny, -tiny, tiny / 8, 1e-45, mx, -mx, mx / 2,
                     np.nextafter(f32(1.0), f32(2.0)), 3.0e38, 2.0 ** -24, 1.0 + 2.0 ** -23], f32)
    a, b = np.meshgrid(vals, vals)
    _check(a.ravel(), b.ravel())
