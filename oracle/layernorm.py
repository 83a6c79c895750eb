"""LayerNorm of the rows of X, the step before the QKV and MLP-up Fprop.

Test infrastructure (see ``oracle/__init__``).

y[r, c] = (x[r, c] - mu_r) * rsigma_r * gamma[c] + beta[c], with mu_r the mean of
row r, var_r its (biased) variance and rsigma_r = 1 / sqrt(var_r + eps): the
te.LayerNorm module that Transformer Engine fuses with the quantization of its
output ("Introduction to FP8 training using Transformer Engine", the module list
and fused kernels of the introduction and of section "Transformer Engine の使い方").
Plain fp64 definition; parity pinned by closed forms, invariances and loops
(tests/test_oracle_layernorm).
"""
from __future__ import annotations

import numpy as np


def layernorm(x, gamma, beta, eps: float):
    """(y [R, C], mu [R], rsigma [R]) in fp64."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=1)
    var = ((x - mu[:, None]) ** 2).mean(axis=1)
    rsigma = 1.0 / np.sqrt(var + float(eps))
    y = (x - mu[:, None]) * rsigma[:, None] * np.asarray(gamma, np.float64)[None, :] + \
        np.asarray(beta, np.float64)[None, :]
    return y, mu, rsigma
