"""fp64 GEMM over dequantized operands, with the linear layer's epilogue.

Test infrastructure (see ``oracle/__init__``).

Every GEMM of the path is D[m, n] = alpha * sum_k A[m, k] * B[n, k] (+ bias[n]),
with A [M, K] and B [N, K] both stored contraction-major.  For a linear layer
Y = X W^T + b ("Introduction to FP8 training using Transformer Engine", section
"Transformer Engine の使い方": ``te.Linear(768, 768, bias=True)``):
  Fprop  Y  = X  W^T     A = X row copy,  B = W row copy         (M x N_out x K_in)
  Dgrad  dX = dY W       A = dY row copy, B = W col copy         (M x K_in x N_out)
  Wgrad  dW = dY^T X     A = dY col copy, B = X col copy         (N_out x K_in x M)
("How to Optimize Transformer-Based Models for Low-Precision Training", section
"autocast モードの使用と事前量子化の比較": Fprop, Dgrad and Wgrad shapes benchmarked
separately).  The product is taken in fp64 (numpy matmul serves as the
library primitive for the contraction).  Parity: pinned by brute-force loops
on tiny shapes and exact small-integer products (tests/test_oracle_gemm).
"""
from __future__ import annotations

import numpy as np


def gemm(a_deq, b_deq, alpha: float = 1.0, bias=None) -> np.ndarray:
    """D = alpha * A @ B^T (+ bias broadcast over rows), all fp64."""
    a = np.asarray(a_deq, dtype=np.float64)
    b = np.asarray(b_deq, dtype=np.float64)
    assert a.shape[1] == b.shape[1]
    d = (a @ b.T) * float(alpha)
    if bias is not None:
        d = d + np.asarray(bias, dtype=np.float64)[None, :]
    return d


def gemm_accumulate(d_old, a_deq, b_deq, alpha: float = 1.0, bias=None) -> np.ndarray:
    """Wgrad accumulated into an fp32 main gradient: D_new = D_old + alpha * A @ B^T (+ bias).

    The weight gradient of successive micro-batches is summed into one fp32 buffer
    (the NeMo ``fp8_wgrad`` key of "Introduction to FP8 training using Transformer
    Engine", section "Transformer Engine 統合済みライブラリの利用").  fp64 here; the
    device adds once per element in fp32.
    """
    return np.asarray(d_old, dtype=np.float64) + gemm(a_deq, b_deq, alpha, bias)


def linear_shapes(hidden: int, ffn: int, tokens: int):
    """The 12 GEMM shapes (name, pass, M, N, K) of one transformer layer's linears.

    Linears (in -> out): QKV h -> 3h, attention output h -> h, MLP up h -> f,
    MLP down f -> h; per linear Fprop (M=tokens, N=out, K=in), Dgrad
    (M=tokens, N=in, K=out) and Wgrad (M=out, N=in, K=tokens).  ("How to
    Optimize Transformer-Based Models for Low-Precision Training", sections
    "モデル設定とトレーニング入力" and "autocast モードの使用と事前量子化の比較":
    M = micro_batch * seq_len, 12 GEMM shapes.)
    """
    linears = [("qkv", hidden, 3 * hidden), ("attn_out", hidden, hidden),
               ("mlp_up", hidden, ffn), ("mlp_down", ffn, hidden)]
    out = []
    for name, k_in, n_out in linears:
        out.append((name, "fprop", tokens, n_out, k_in))
        out.append((name, "dgrad", tokens, k_in, n_out))
        out.append((name, "wgrad", n_out, k_in, tokens))
    return out


def rel_frobenius(d, ref) -> float:
    d = np.asarray(d, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(d - ref) / (den if den > 0 else 1.0))
