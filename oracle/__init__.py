"""CPU oracle for the quantized-linear hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the hot path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import it.  The product library never calls it
and shares no code with it; the two meet only through the seeded input
generators in ``synthetic/``.

Precision: every step that decides an integer (a quantized code, a block
scale byte) is taken in IEEE fp32 with round-to-nearest-even, the precision the
kernels use (the pages fix none).  GEMM reference products are taken in fp64.

Modules
  formats   -- E4M3 / E5M2 / E2M1 / UE4M3 / E8M0 encoders and decoders
  philox    -- Philox4x32-10 counter-based generator (Salmon et al., SC'11)
  recipes   -- DelayedScaling and CurrentScaling scale updates
  quantize  -- per-tensor FP8, MXFP8 and NVFP4 quantizers (RHT, SR, 2D)
  gemm      -- fp64 GEMM over dequantized operands, epilogue, Wgrad accumulation
  layernorm -- LayerNorm of the rows (the step before the QKV / MLP-up Fprop)

Every function is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*``
to a closed form, a brute-force check, a hand-worked table or an independent
second implementation.  Parity status per function is listed in each module's
docstring; none is unpinned.
"""
from . import formats, philox, recipes, quantize, gemm, layernorm  # noqa: F401
