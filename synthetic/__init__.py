"""Seeded synthetic inputs shared by the tests, the bench and the oracle.

This module holds no arithmetic of the quantized-linear method: it only draws
random tensors with the value distributions of the workloads and hands them to
either side (the CUDA library through its binding, the CPU oracle directly).

Workloads (shapes from "How to Optimize Transformer-Based Models for
Low-Precision Training", section "モデル設定とトレーニング入力": CodonFM-5B,
hidden 4096, intermediate 16384, micro-batch 31, sequence 512 -> M = 15872
tokens; the single linear from "Introduction to FP8 training using Transformer
Engine", section "Transformer Engine の使い方": te.Linear(768, 768) on a
1024 x 768 input drawn with torch.rand):

  linear768   X [1024, 768] fp32 ~ U[0, 1), W [768, 768] ~ N(0, 0.02^2),
              bias [768] ~ N(0, 0.02^2), dY [1024, 768] ~ N(0, 1e-3^2)
  codonfm     bf16 X ~ N(0, 1), W ~ N(0, 0.02^2), dY ~ N(0, 1e-3^2)
  heavy-tail  bf16 X ~ Student-t(nu = 3) with 0.1 % of positions scaled x100

No dataset is involved: CodonFM-5B contributes only its layer sizes.
"""
from __future__ import annotations

import torch

HIDDEN = 4096
FFN = 16384
TOKENS = 31 * 512  # micro_batch_size * sequence_length = 15872


def seed_for(config: int, linear: int, tensor: int, base: int = 1234) -> int:
    """Fixed seed recipe: base + 1000*config + 10*linear + tensor."""
    return base + 1000 * config + 10 * linear + tensor


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(shape, std: float, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 and rounded to ``dtype``."""
    t = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return (t * std).to(dtype)


def uniform(shape, seed: int, dtype=torch.float32, device="cpu") -> torch.Tensor:
    """U[0, 1) (torch.rand) in ``dtype``."""
    return torch.rand(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32).to(dtype)


def student_t_outliers(shape, seed: int, nu: float = 3.0, frac: float = 1e-3, factor: float = 100.0,
                       dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Student-t(nu) values with a seeded fraction ``frac`` of positions scaled by ``factor``.

    t = Z / sqrt(V / nu) with Z ~ N(0, 1) and V ~ chi^2(nu) = 2 * Gamma(nu / 2).
    """
    g = _gen(seed, device)
    z = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    conc = torch.full(shape, nu / 2.0, device=device, dtype=torch.float32)
    # torch's Gamma sampler takes no generator; fork the global state under the seed instead
    with torch.random.fork_rng(devices=[] if device == "cpu" else [torch.device(device)]):
        torch.manual_seed(int(seed) + 7)
        v = torch._standard_gamma(conc) * 2.0
    t = z / torch.sqrt(v / nu)
    mask = torch.rand(*shape, generator=g, device=device) < frac
    t = torch.where(mask, t * factor, t)
    return t.to(dtype)


def rht_sign_mask(seed: int) -> int:
    """16 random sign bits for the random Hadamard transform (bit j set -> column j negated)."""
    return int(torch.randint(0, 1 << 16, (1,), generator=_gen(seed)).item())


def linear768(step: int, base: int = 1234):
    """Inputs of the single 768 -> 768 linear at a given step (X re-drawn every step)."""
    x = uniform((1024, 768), seed=base + step)
    w = gaussian((768, 768), 0.02, seed=base + 100, dtype=torch.float32)
    b = gaussian((768,), 0.02, seed=base + 101, dtype=torch.float32)
    dy = gaussian((1024, 768), 1e-3, seed=base + 200 + step, dtype=torch.float32)
    return x, w, b, dy


def layer_linears(hidden: int = HIDDEN, ffn: int = FFN):
    """(name, in_features, out_features) of the four linears of one layer."""
    return [("qkv", hidden, 3 * hidden), ("attn_out", hidden, hidden),
            ("mlp_up", hidden, ffn), ("mlp_down", ffn, hidden)]


def codonfm_linear(idx: int, tokens: int = TOKENS, hidden: int = HIDDEN, ffn: int = FFN,
                   config: int = 2, device="cpu", heavy_tail: bool = False):
    """(X [tokens, in], W [out, in], dY [tokens, out]) bf16 for linear ``idx`` of a layer."""
    _, k_in, n_out = layer_linears(hidden, ffn)[idx]
    sx, sw, sd = (seed_for(config, idx, t) for t in range(3))
    if heavy_tail:
        x = student_t_outliers((tokens, k_in), sx, device=device)
    else:
        x = gaussian((tokens, k_in), 1.0, sx, device=device)
    w = gaussian((n_out, k_in), 0.02, sw, device=device)
    dy = gaussian((tokens, n_out), 1e-3, sd, device=device)
    return x, w, dy


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor (what the oracle consumes)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
