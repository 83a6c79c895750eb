"""Scaling recipes: DelayedScaling (amax history) and CurrentScaling.

Test infrastructure (see ``oracle/__init__``).

Sources.  Every tensor (weights and activations) carries its own scaling
factor, refreshed every step because ranges move during training ("Introduction
to FP8 training using Transformer Engine", section "FP8 Training について").
The recipe holds the format, the history length and the algorithm that turns
the history into an amax (same page, section "Transformer Engine の使い方":
``DelayedScaling(fp8_format=Format.HYBRID, amax_history_len=16,
amax_compute_algo="max")``), plus a margin and an update interval (same page,
NeMo keys ``fp8_margin``, ``fp8_interval``, ``fp8_amax_history_len``,
``fp8_amax_compute_algo`` = 'max' | 'most_recent').  DelayedScaling quantizes
with a scale derived from past amaxes; CurrentScaling from the tensor's own
amax ("How to Optimize Transformer-Based Models for Low-Precision Training",
section "autocast モードの使用と事前量子化の比較").

Readings where the pages are silent:
  * initial state: history all zeros, scale 1, scale_inv 1;
  * step t quantizes with the current scale, then records its amax a_t into
    slot t mod L, then (if (t+1) mod interval == 0) recomputes the scale;
  * scale = fl32(fl32(fmax / amax) * 2**-margin); kept unchanged when amax is
    zero or not finite, or when the new scale is not finite;
  * scale_inv = fl32(1 / scale);
  * CurrentScaling: scale = fl32(fmax / a) for a > 0 with a finite result,
    else 1; no margin.
All arithmetic fp32.  Parity: pinned (hand-worked tables, tests/test_oracle_recipes).
"""
from __future__ import annotations

import numpy as np

from .formats import FMAX

ALGO_MAX = 0
ALGO_MOST_RECENT = 1

f32 = np.float32


def _scale_from_amax(fmax: float, amax: np.float32, margin: int, old: np.float32) -> np.float32:
    amax = f32(amax)
    if not (np.isfinite(amax) and amax > 0):
        return f32(old)
    with np.errstate(over="ignore", divide="ignore"):
        s = f32(f32(fmax) / amax)
        s = f32(s * f32(2.0 ** (-margin)))
    if not np.isfinite(s):
        return f32(old)
    return s


class DelayedScalingState:
    """State of one tensor role under DelayedScaling (history ring + scale)."""

    def __init__(self, fmt: str, history_len: int, algo: int = ALGO_MAX, margin: int = 0,
                 interval: int = 1):
        assert history_len >= 1 and interval >= 1
        self.fmt, self.L, self.algo, self.margin, self.interval = fmt, history_len, algo, margin, interval
        self.hist = np.zeros(history_len, dtype=np.float32)
        self.scale = f32(1.0)
        self.scale_inv = f32(1.0)

    def update(self, amax_t, step: int) -> None:
        """Record the amax observed at ``step`` and refresh the scale."""
        a = f32(amax_t)
        self.hist[step % self.L] = a
        if (step + 1) % self.interval != 0:
            return
        if self.algo == ALGO_MAX:
            eff = f32(np.max(self.hist))
        else:
            eff = a
        self.scale = _scale_from_amax(FMAX[self.fmt], eff, self.margin, self.scale)
        self.scale_inv = f32(f32(1.0) / self.scale)


def current_scale(amax, fmt: str):
    """CurrentScaling: (scale, scale_inv) from the tensor's own amax."""
    s = _scale_from_amax(FMAX[fmt], f32(amax), 0, f32(1.0))
    return s, f32(f32(1.0) / s)
