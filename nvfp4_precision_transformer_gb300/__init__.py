"""GB300-native quantized linear-layer hot path (FP8 / MXFP8 / NVFP4, tcgen05 GEMMs).

The compute lives in ``libte_gb300.so`` (hand-written CUDA for sm_103a behind
the C ABI in ``include/te_gb300.h``); this package is the thin Python side:
``_lib`` binds the C entry points by name, ``linear`` composes them into the
per-recipe linear-layer steps (Fprop / Dgrad / Wgrad) and ``shapes`` derives
the GEMM shapes of a transformer layer from its configuration.
"""
from ._lib import (  # noqa: F401
    ALGO_MAX, ALGO_MOST_RECENT, BF16, K_MAJOR, MN_MAJOR, E2M1, E4M3, E5M2, E8M0, F32, NVFP4_2D, NVFP4_RHT_COL, NVFP4_SR, UE4M3,
    TEError, te_amax_reduce, te_dbias_workspace_bytes, te_gemm_bf16, te_gemm_fp8, te_gemm_mxfp8, te_gemm_nvfp4, te_get_last_error, te_layernorm_fp8,
    te_launch_count, te_quantize_fp8, te_quantize_fp8_dbias, te_quantize_fp8_dbias_noalloc, te_quantize_mxfp8, te_quantize_nvfp4, te_recipe, te_scale_bytes,
    te_scale_unswizzle, te_scale_update, te_selftest_wait_timeout, te_status_str, lib,
)
