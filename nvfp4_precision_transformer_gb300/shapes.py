"""GEMM shapes of one transformer layer derived from its configuration.

"How to Optimize Transformer-Based Models for Low-Precision Training",
sections "モデル設定とトレーニング入力" and "autocast モードの使用と事前量子化の比較":
the benchmark tool turns (hidden, intermediate, micro-batch, sequence length)
into M = micro_batch * seq_len tokens and the 12 GEMMs of a layer -- four
linears (QKV, attention output, MLP up, MLP down) times Fprop, Dgrad, Wgrad,
each benchmarked separately because the aspect ratios differ.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class LayerConfig:
    hidden: int = 4096
    intermediate: int = 16384
    heads: int = 32
    layers: int = 24
    micro_batch: int = 31
    seq_len: int = 512

    @property
    def tokens(self) -> int:
        return self.micro_batch * self.seq_len


@dataclass(frozen=True)
class Gemm:
    linear: str
    pass_: str   # fprop | dgrad | wgrad
    M: int
    N: int
    K: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def linears(cfg: LayerConfig):
    """(name, in_features, out_features) of the layer's four linears."""
    h, f = cfg.hidden, cfg.intermediate
    return [("qkv", h, 3 * h), ("attn_out", h, h), ("mlp_up", h, f), ("mlp_down", f, h)]


def layer_gemms(cfg: LayerConfig):
    out = []
    for name, k_in, n_out in linears(cfg):
        out.append(Gemm(name, "fprop", cfg.tokens, n_out, k_in))     # Y  = X W^T
        out.append(Gemm(name, "dgrad", cfg.tokens, k_in, n_out))     # dX = dY W
        out.append(Gemm(name, "wgrad", n_out, k_in, cfg.tokens))     # dW = dY^T X
    return out


def layer_flops(cfg: LayerConfig) -> int:
    return sum(g.flops for g in layer_gemms(cfg))
