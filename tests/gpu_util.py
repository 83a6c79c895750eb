"""Helpers shared by the GPU parity tests: run the library on torch tensors and
bring results back as numpy arrays in the oracle's logical layouts."""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_precision_transformer_gb300 as te
from oracle import formats as F
from synthetic import bf16_bits

DEV = "cuda"


def f32_np(x: torch.Tensor) -> np.ndarray:
    """Exact fp32 numpy view of a bf16 / fp32 tensor (what the oracle consumes)."""
    if x.dtype == torch.bfloat16:
        return F.bf16_bits_to_f32(bf16_bits(x))
    return x.detach().cpu().float().numpy()


def scalar(v=0.0) -> torch.Tensor:
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def u8(*shape) -> torch.Tensor:
    return torch.full(shape, 0xA5, dtype=torch.uint8, device=DEV)   # poison: unwritten bytes show up


def check_no_device_error():
    st = te.te_get_last_error()
    assert st == 0, te.te_status_str(st)


def fp8(x, fmt, scale=None, current=False, row=True, col=True):
    R, C = x.shape
    q_row = u8(R, C) if row else None
    q_col = u8(C, R) if col else None
    amax, sinv = scalar(-1.0), scalar(-1.0)
    sc = scalar(scale) if scale is not None else None
    te.te_quantize_fp8(x, fmt, scale=sc, compute_scale=int(current), q_row=q_row, q_col=q_col,
                       amax_out=amax, scale_inv_out=sinv)
    torch.cuda.synchronize()
    return (q_row.cpu().numpy() if row else None, q_col.cpu().numpy() if col else None,
            np.float32(amax.item()), np.float32(sinv.item()))


def mxfp8(x, row=True, col=True):
    R, C = x.shape
    out = {}
    q_row = u8(R, C) if row else None
    s_row = u8(te.te_scale_bytes(te.E8M0, R, C)) if row else None
    q_col = u8(C, R) if col else None
    s_col = u8(te.te_scale_bytes(te.E8M0, C, R)) if col else None
    te.te_quantize_mxfp8(x, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    if row:
        out["q_row"] = q_row.cpu().numpy()
        out["s_row_raw"] = s_row.cpu().numpy()
        out["s_row"] = te.te_scale_unswizzle(te.E8M0, R, C, out["s_row_raw"])
    if col:
        out["q_col"] = q_col.cpu().numpy()
        out["s_col_raw"] = s_col.cpu().numpy()
        out["s_col"] = te.te_scale_unswizzle(te.E8M0, C, R, out["s_col_raw"])
    return out


def amax(x, rht_signs=None):
    a = scalar(-1.0)
    ar = scalar(-1.0) if rht_signs is not None else None
    te.te_amax_reduce(x, a, ar, rht_signs or 0)
    torch.cuda.synchronize()
    return np.float32(a.item()), (np.float32(ar.item()) if ar is not None else None)


def nvfp4(x, flags=0, signs=0, seed=0, offset=0, row=True, col=True):
    """Returns dict with unpacked codes [.., cols] (nibbles), logical scales, gdec and raw buffers."""
    R, C = x.shape
    a, ar = scalar(), scalar()
    te.te_amax_reduce(x, a, ar if col and (flags & te.NVFP4_RHT_COL) else None, signs)
    q_row = u8(R, C // 2) if row else None
    s_row = u8(te.te_scale_bytes(te.UE4M3, R, C)) if row else None
    g_row = scalar(-1.0) if row else None
    q_col = u8(C, R // 2) if col else None
    s_col = u8(te.te_scale_bytes(te.UE4M3, C, R)) if col else None
    g_col = scalar(-1.0) if col else None
    te.te_quantize_nvfp4(x, flags, signs, seed, offset, a, ar, q_row, s_row, g_row, q_col, s_col, g_col)
    torch.cuda.synchronize()
    out = {"amax": np.float32(a.item()), "amax_rht": np.float32(ar.item())}
    if row:
        out["q_row_packed"] = q_row.cpu().numpy()
        out["q_row"] = unpack_e2m1(out["q_row_packed"])
        out["s_row_raw"] = s_row.cpu().numpy()
        out["s_row"] = te.te_scale_unswizzle(te.UE4M3, R, C, out["s_row_raw"])
        out["g_row"] = np.float32(g_row.item())
    if col:
        out["q_col_packed"] = q_col.cpu().numpy()
        out["q_col"] = unpack_e2m1(out["q_col_packed"])
        out["s_col_raw"] = s_col.cpu().numpy()
        out["s_col"] = te.te_scale_unswizzle(te.UE4M3, C, R, out["s_col_raw"])
        out["g_col"] = np.float32(g_col.item())
    return out


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Split packed E2M1 bytes into nibbles (element 2i = low nibble)."""
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def assert_equal_codes(got, exp, what=""):
    got = np.asarray(got)
    exp = np.asarray(exp)
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:4].tolist()}: " \
                          f"got {[int(got[tuple(b)]) for b in bad[:4]]} exp {[int(exp[tuple(b)]) for b in bad[:4]]}"


# ---- GEMM parity bar ---------------------------------------------------------------------------

GEMM_TOL = 1e-3


def ulp(x, precision_bits: int) -> np.ndarray:
    """One unit in the last place of |x| in a binary format with ``precision_bits`` significand
    bits (24 fp32, 8 bf16), normal range (the exponent is floored at -126)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.exp2(e - (precision_bits - 1))


def check_gemm(got, a64, b64, bias=None, bf16_out=False, what="", tol=GEMM_TOL):
    """The GEMM parity bar on D = A B^T (+ bias) against the oracle's fp64 product of its own
    dequantized operands a64 [m, K], b64 [n, K] (``got`` [m, n], the device's outputs widened):

    * relative Frobenius error <= tol: fp32 outputs against the fp64 product, bf16 outputs
      against the bf16-rounded fp64 product (bf16 rounding alone is ~1.7e-3 on Gaussian data);
    * every element within K * 2^-23 * sum_k |a_k b_k| (fp32 accumulation over K terms) plus
      one output ulp of the product (the epilogue's rounding), so that a few wrong elements
      cannot hide under the norm.
    Returns (rel-Frobenius, largest |error| / bound)."""
    from oracle import formats as F
    from oracle import gemm as OG
    a64 = np.asarray(a64, np.float64)
    b64 = np.asarray(b64, np.float64)
    got = np.asarray(got, np.float64)
    ref = OG.gemm(a64, b64, bias=bias)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    exp = F.bf16_bits_to_f32(F.f64_to_bf16_bits(ref)).astype(np.float64) if bf16_out else ref
    err = OG.rel_frobenius(got, exp)
    K = a64.shape[1]
    S = np.abs(a64) @ np.abs(b64).T
    bound = K * 2.0 ** -23 * S + ulp(ref, 8 if bf16_out else 24)
    ratio = np.abs(got - ref) / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    assert err <= tol, f"{what}: rel-Frobenius {err:.3e}"
    if worst > 1.0:
        i = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        raise AssertionError(f"{what}: element {i} off by {abs(got[i] - ref[i]):.3e} > bound {bound[i]:.3e} "
                             f"({int(np.sum(ratio > 1))} elements out of bound)")
    return err, worst
