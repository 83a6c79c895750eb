"""ctypes binding of libte_gb300.so (argument marshalling only).

Every function here has the name of the C entry point it wraps and does no
arithmetic of its own: it turns torch tensors into device pointers and sizes,
passes the current CUDA stream, and raises TEError on a non-zero status.  The
library must have been built (``build.build()``); importing this module fails
loudly otherwise -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libte_gb300.so")

# te_dtype
F32, BF16, E4M3, E5M2, E2M1, E8M0, UE4M3 = range(7)
# NVFP4 flags
NVFP4_2D, NVFP4_RHT_COL, NVFP4_SR = 1, 2, 4
ALGO_MAX, ALGO_MOST_RECENT = 0, 1
# te_layout
K_MAJOR, MN_MAJOR = 0, 1

STATUS = {0: "TE_OK", 1: "TE_ERR_NULL", 2: "TE_ERR_SHAPE", 3: "TE_ERR_ALIGN", 4: "TE_ERR_DTYPE",
          5: "TE_ERR_UNSUPPORTED", 6: "TE_ERR_CUDA", 7: "TE_ERR_TIMEOUT", 8: "TE_ERR_ARG"}

# exported symbols and their signatures (restype, argtypes)
_vp, _i64, _u32, _u64, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int
_st = ctypes.c_int


class te_recipe(ctypes.Structure):
    _fields_ = [("fwd_fmt", ctypes.c_int), ("bwd_fmt", ctypes.c_int), ("amax_history_len", ctypes.c_int),
                ("amax_compute_algo", ctypes.c_int), ("margin", ctypes.c_int), ("interval", ctypes.c_int)]


SIGNATURES = {
    "te_amax_reduce": (_st, [_vp, _int, _i64, _i64, _vp, _vp, _u32, _vp]),
    "te_scale_update": (_st, [ctypes.POINTER(te_recipe), _int, _int, _vp, _vp, _vp, _vp, _i64, _vp]),
    "te_quantize_fp8": (_st, [_vp, _int, _i64, _i64, _int, _vp, _int, _vp, _vp, _vp, _vp, _vp]),
    "te_quantize_mxfp8": (_st, [_vp, _int, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "te_layernorm_fp8": (_st, [_vp, _int, _i64, _i64, _vp, _vp, ctypes.c_float, _int, _vp, _vp, _vp, _vp, _vp, _vp,
                               _vp, _vp]),
    "te_quantize_fp8_dbias_noalloc": (_st, [_vp, _int, _i64, _i64, _int, _vp, _int, _vp, _vp, _vp, _vp, _vp, _vp]),
    "te_dbias_workspace_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "te_quantize_fp8_dbias": (_st, [_vp, _int, _i64, _i64, _int, _vp, _int, _vp, _vp, _vp, _vp, _vp, _vp,
                                    ctypes.c_size_t, _vp]),
    "te_quantize_nvfp4": (_st, [_vp, _int, _i64, _i64, _u32, _u32, _u64, _u64, _vp, _vp,
                                _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "te_gemm_bf16": (_st, [_vp, _int, _vp, _int, _vp, _vp, _int, _int, _i64, _i64, _i64, _vp]),
    "te_gemm_fp8": (_st, [_vp, _int, _vp, _int, _vp, _vp, _vp, _vp, _int, _int, _i64, _i64, _i64, _vp]),
    "te_gemm_mxfp8": (_st, [_vp, _int, _vp, _vp, _int, _vp, _vp, _vp, _int, _int, _i64, _i64, _i64, _vp]),
    "te_gemm_nvfp4": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _i64, _i64, _i64, _vp]),
    "te_scale_bytes": (ctypes.c_size_t, [_int, _i64, _i64]),
    "te_scale_unswizzle": (_st, [_int, _i64, _i64, _vp, _vp]),
    "te_status_str": (ctypes.c_char_p, [_int]),
    "te_get_last_error": (_st, []),
    "te_launch_count": (_u64, []),
    "te_selftest_wait_timeout": (_st, [_vp]),
}


class TEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with nvfp4_precision_transformer_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def _check(name: str, status: int) -> None:
    if status != 0:
        raise TEError(name, status)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _in_dtype(x):
    import torch
    if x.dtype == torch.bfloat16:
        return BF16
    if x.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported input dtype {x.dtype}")


def _rc(x):
    assert x.dim() == 2 and x.is_contiguous()
    return x.shape[0], x.shape[1]


# ---- entry points (same names as the C ABI) ----------------------------------------

def te_amax_reduce(x, amax, amax_rht=None, rht_signs: int = 0, stream=None):
    r, c = _rc(x)
    _check("te_amax_reduce", lib().te_amax_reduce(_ptr(x), _in_dtype(x), r, c, _ptr(amax), _ptr(amax_rht),
                                                  rht_signs & 0xFFFFFFFF, _stream(stream)))


def te_scale_update(recipe: te_recipe, is_backward: int, hist, amax, scale, scale_inv, step: int, stream=None):
    n = amax.numel()
    _check("te_scale_update", lib().te_scale_update(ctypes.byref(recipe), int(is_backward), n, _ptr(hist),
                                                    _ptr(amax), _ptr(scale), _ptr(scale_inv), int(step),
                                                    _stream(stream)))


def te_quantize_fp8(x, fmt: int, scale=None, compute_scale: int = 0, q_row=None, q_col=None, amax_out=None,
                    scale_inv_out=None, stream=None):
    r, c = _rc(x)
    _check("te_quantize_fp8", lib().te_quantize_fp8(_ptr(x), _in_dtype(x), r, c, fmt, _ptr(scale), compute_scale,
                                                    _ptr(q_row), _ptr(q_col), _ptr(amax_out), _ptr(scale_inv_out),
                                                    _stream(stream)))


def te_dbias_workspace_bytes(rows: int, cols: int) -> int:
    return int(lib().te_dbias_workspace_bytes(rows, cols))


def te_quantize_fp8_dbias(x, fmt: int, dbias, workspace, scale=None, compute_scale: int = 0, q_row=None, q_col=None,
                          amax_out=None, scale_inv_out=None, stream=None):
    r, c = _rc(x)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("te_quantize_fp8_dbias", lib().te_quantize_fp8_dbias(
        _ptr(x), _in_dtype(x), r, c, fmt, _ptr(scale), compute_scale, _ptr(q_row), _ptr(q_col), _ptr(amax_out),
        _ptr(scale_inv_out), _ptr(dbias), _ptr(workspace), nbytes, _stream(stream)))


def te_quantize_fp8_dbias_noalloc(x, fmt: int, dbias, scale=None, compute_scale: int = 0, q_row=None, q_col=None,
                                  amax_out=None, scale_inv_out=None, stream=None):
    """te_quantize_fp8_dbias with the library's fixed scratch array instead of a workspace."""
    r, c = _rc(x)
    _check("te_quantize_fp8_dbias_noalloc", lib().te_quantize_fp8_dbias_noalloc(
        _ptr(x), _in_dtype(x), r, c, fmt, _ptr(scale), compute_scale, _ptr(q_row), _ptr(q_col), _ptr(amax_out),
        _ptr(scale_inv_out), _ptr(dbias), _stream(stream)))


def te_layernorm_fp8(x, gamma, beta, eps: float, fmt: int, scale, q_row, ln_out=None, mu=None, rsigma=None,
                     amax_out=None, scale_inv_out=None, stream=None):
    r, c = _rc(x)
    _check("te_layernorm_fp8", lib().te_layernorm_fp8(
        _ptr(x), _in_dtype(x), r, c, _ptr(gamma), _ptr(beta), float(eps), fmt, _ptr(scale), _ptr(q_row),
        _ptr(ln_out), _ptr(mu), _ptr(rsigma), _ptr(amax_out), _ptr(scale_inv_out), _stream(stream)))


def te_quantize_mxfp8(x, q_row=None, s_row=None, q_col=None, s_col=None, stream=None):
    r, c = _rc(x)
    _check("te_quantize_mxfp8", lib().te_quantize_mxfp8(_ptr(x), _in_dtype(x), r, c, _ptr(q_row), _ptr(s_row),
                                                        _ptr(q_col), _ptr(s_col), _stream(stream)))


def te_quantize_nvfp4(x, flags: int = 0, rht_signs: int = 0, seed: int = 0, offset: int = 0, amax=None,
                      amax_rht=None, q_row=None, s_row=None, gdec_row=None, q_col=None, s_col=None, gdec_col=None,
                      stream=None):
    r, c = _rc(x)
    _check("te_quantize_nvfp4", lib().te_quantize_nvfp4(_ptr(x), _in_dtype(x), r, c, flags, rht_signs, seed,
                                                        offset, _ptr(amax), _ptr(amax_rht), _ptr(q_row),
                                                        _ptr(s_row), _ptr(gdec_row), _ptr(q_col), _ptr(s_col),
                                                        _ptr(gdec_col), _stream(stream)))


def _out_dtype(d):
    import torch
    if d.dtype == torch.bfloat16:
        return BF16
    if d.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported output dtype {d.dtype}")


# accumulate=1: D (fp32) += the GEMM's result instead of D = result (Wgrad into a main
# gradient); the library rejects it for a bf16 D.

def te_gemm_bf16(A, B, D, bias=None, a_layout: int = 0, b_layout: int = 0, accumulate: int = 0, stream=None):
    """A is [M, K] (K_MAJOR) or [K, M] (MN_MAJOR); B is [N, K] or [K, N]; D is [M, N]."""
    M, N = D.shape
    K = A.shape[1] if a_layout == K_MAJOR else A.shape[0]
    _check("te_gemm_bf16", lib().te_gemm_bf16(_ptr(A), a_layout, _ptr(B), b_layout, _ptr(bias), _ptr(D),
                                              _out_dtype(D), int(accumulate), M, N, K, _stream(stream)))


def te_gemm_fp8(A, fa: int, B, fb: int, a_scale_inv, b_scale_inv, D, bias=None, accumulate: int = 0, stream=None):
    M, K = A.shape
    N = B.shape[0]
    _check("te_gemm_fp8", lib().te_gemm_fp8(_ptr(A), fa, _ptr(B), fb, _ptr(a_scale_inv), _ptr(b_scale_inv),
                                            _ptr(bias), _ptr(D), _out_dtype(D), int(accumulate), M, N, K,
                                            _stream(stream)))


def te_gemm_mxfp8(A, sA, B, sB, D, bias=None, fa: int = E4M3, fb: int = E4M3, accumulate: int = 0, stream=None):
    M, K = A.shape
    N = B.shape[0]
    _check("te_gemm_mxfp8", lib().te_gemm_mxfp8(_ptr(A), fa, _ptr(sA), _ptr(B), fb, _ptr(sB), _ptr(bias), _ptr(D),
                                                _out_dtype(D), int(accumulate), M, N, K, _stream(stream)))


def te_gemm_nvfp4(A, sA, gA, B, sB, gB, D, bias=None, accumulate: int = 0, stream=None):
    M, Kh = A.shape
    N = B.shape[0]
    _check("te_gemm_nvfp4", lib().te_gemm_nvfp4(_ptr(A), _ptr(sA), _ptr(gA), _ptr(B), _ptr(sB), _ptr(gB),
                                                _ptr(bias), _ptr(D), _out_dtype(D), int(accumulate), M, N, 2 * Kh,
                                                _stream(stream)))


def te_scale_bytes(scale_fmt: int, rows: int, cols: int) -> int:
    return int(lib().te_scale_bytes(scale_fmt, rows, cols))


def te_scale_unswizzle(scale_fmt: int, rows: int, cols: int, swizzled: np.ndarray) -> np.ndarray:
    blk = 32 if scale_fmt == E8M0 else 16
    sw = np.ascontiguousarray(swizzled, dtype=np.uint8)
    out = np.zeros((rows, cols // blk), dtype=np.uint8)
    _check("te_scale_unswizzle", lib().te_scale_unswizzle(scale_fmt, rows, cols, sw.ctypes.data,
                                                          out.ctypes.data))
    return out


def te_status_str(status: int) -> str:
    return lib().te_status_str(status).decode()


def te_get_last_error() -> int:
    return int(lib().te_get_last_error())


def te_launch_count() -> int:
    return int(lib().te_launch_count())


def te_selftest_wait_timeout(stream=None):
    _check("te_selftest_wait_timeout", lib().te_selftest_wait_timeout(_stream(stream)))
