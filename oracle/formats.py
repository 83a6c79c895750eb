"""Narrow floating-point formats: encoders (fp32 -> code) and decoders.

Test infrastructure (see ``oracle/__init__``).

The pages only name the formats: FP8 with E4M3 for the forward pass and E5M2
for gradients under ``Format.HYBRID`` ("Introduction to FP8 training using
Transformer Engine", section "Transformer Engine の使い方", recipe example),
MXFP8 and NVFP4 on Blackwell ("transformerengine" repository summary).  The
bit-level definitions used here are the public OCP 8-bit floating point
specification (OFP8: E4M3 bias 7, no infinities, S.1111.111 is NaN, max 448;
E5M2 bias 15, IEEE-like infinities, max 57344) and the OCP Microscaling v1.0
specification (E2M1 bias 1, max 6, no specials; E8M0 = 2**(b-127), 0xFF NaN).
UE4M3 is E4M3 with the sign bit fixed at 0 (the NVFP4 block scale).

Reading of rounding: round-to-nearest, ties to even, subnormals included,
then saturate: any finite or infinite magnitude above the format's largest
finite value becomes +-max ("satfinite").  NaN maps to the NaN code 0x7F with
the input's sign for E4M3 / E5M2; NaN is outside the contract for E2M1.
Zero keeps its sign (-0 -> 0x80 for FP8, 0x8 for E2M1).

Two independent encoders are provided:
  * ``encode``       -- integer rounding of the fp32 significand (bit method)
  * ``encode_table`` -- nearest decoded value by binary search over the code
                        table, ties to the even code (table method)
They share only the format parameters.  Parity: pinned (tests/test_oracle_formats).
"""
from __future__ import annotations

import numpy as np

# (exponent bits, mantissa bits, bias, largest finite magnitude code, NaN code or None)
FORMATS = {
    "e4m3": dict(ebits=4, mbits=3, bias=7, max_code=0x7E, nan_code=0x7F, nbits=8),
    "e5m2": dict(ebits=5, mbits=2, bias=15, max_code=0x7B, nan_code=0x7F, nbits=8),
    "e2m1": dict(ebits=2, mbits=1, bias=1, max_code=0x7, nan_code=None, nbits=4),
}

FMAX = {"e4m3": 448.0, "e5m2": 57344.0, "e2m1": 6.0}


def _f32_bits(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def decode(codes, fmt: str) -> np.ndarray:
    """Value of each code as float64 (NaN / inf where the format has them)."""
    p = FORMATS[fmt]
    c = np.asarray(codes).astype(np.int64)
    nb, mb = p["nbits"], p["mbits"]
    sign = (c >> (nb - 1)) & 1
    mag = c & ((1 << (nb - 1)) - 1)
    e = mag >> mb
    m = mag & ((1 << mb) - 1)
    emin = 1 - p["bias"]
    sub = m.astype(np.float64) * 2.0 ** (emin - mb)
    nrm = (1.0 + m.astype(np.float64) / (1 << mb)) * np.exp2((e - p["bias"]).astype(np.float64))
    val = np.where(e == 0, sub, nrm)
    if fmt == "e4m3":
        val = np.where(mag == 0x7F, np.nan, val)
    elif fmt == "e5m2":
        val = np.where(mag == 0x7C, np.inf, val)
        val = np.where(mag > 0x7C, np.nan, val)
    return np.where(sign == 1, -val, val)


def encode(x, fmt: str) -> np.ndarray:
    """Bit method: round the 24-bit fp32 significand to the target quantum.

    For a normal fp32 value v = S * 2**(e-23) (S = 1.m as a 24-bit integer),
    the target quantum is 2**(max(e, emin) - mbits).  The number of dropped bits
    is d = max(e, emin) - mbits - e + 23; the kept integer R is S >> d rounded
    half-to-even on the dropped remainder.  The magnitude code follows from R
    (subnormal: code = R; normal: code = (e - emin + 1) << mbits + R - 2**mbits,
    which also carries a rounding overflow into the exponent field).
    """
    p = FORMATS[fmt]
    mb, nb = p["mbits"], p["nbits"]
    emin = 1 - p["bias"]
    bits = _f32_bits(x).astype(np.int64)
    sign = (bits >> 31) & 1
    e32 = (bits >> 23) & 0xFF
    m32 = bits & 0x7FFFFF
    e = e32 - 127
    S = m32 | (1 << 23)
    d = np.maximum(e, emin) - mb - e + 23
    d_c = np.clip(d, 1, 40)  # d >= 23 - mbits >= 20 always; the upper clip keeps shifts defined
    R = S >> d_c
    rem = S & ((np.int64(1) << d_c) - 1)
    half = np.int64(1) << (d_c - 1)
    up = (rem > half) | ((rem == half) & ((R & 1) == 1))
    R = R + up.astype(np.int64)
    code = np.where(e >= emin, ((e - emin + 1) << mb) + R - (1 << mb), R)
    code = np.where(d > 40, 0, code)          # far below the smallest subnormal
    code = np.where(e32 == 0, 0, code)        # fp32 zero / subnormal: far below every format's range
    code = np.minimum(code, p["max_code"])     # saturate (covers overflow and +-inf)
    if p["nan_code"] is not None:
        code = np.where((e32 == 0xFF) & (m32 != 0), p["nan_code"], code)
    out = code | (sign << (nb - 1))
    return out.astype(np.uint8)


def _table(fmt: str):
    p = FORMATS[fmt]
    codes = np.arange(p["max_code"] + 1)
    vals = decode(codes, fmt)
    assert np.all(np.diff(vals) > 0)
    return codes, vals


def encode_table(x, fmt: str) -> np.ndarray:
    """Table method: nearest non-negative code by value, ties to the even code."""
    p = FORMATS[fmt]
    codes, vals = _table(fmt)
    x32 = np.asarray(x, dtype=np.float32)
    with np.errstate(invalid="ignore"):
        a = np.abs(x32.astype(np.float64))
    sign = (_f32_bits(x32) >> 31).astype(np.int64)
    fin = np.where(np.isnan(a), 0.0, a)
    hi_idx = np.searchsorted(vals, fin, side="left")        # first value >= a
    hi_idx = np.clip(hi_idx, 0, len(vals) - 1)
    lo_idx = np.clip(hi_idx - 1, 0, len(vals) - 1)
    exact = vals[hi_idx] == fin
    d_lo = fin - vals[lo_idx]
    d_hi = vals[hi_idx] - fin
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi_idx] % 2 == 0))
    idx = np.where(exact, hi_idx, np.where(pick_hi, hi_idx, lo_idx))
    code = codes[idx]
    code = np.where(fin > vals[-1], p["max_code"], code)     # saturate
    if p["nan_code"] is not None:
        code = np.where(np.isnan(a), p["nan_code"], code)
    out = code | (sign << (p["nbits"] - 1))
    return out.astype(np.uint8)


def quantize_value(x, fmt: str) -> np.ndarray:
    """fp32 value of the encoded code (what the tensor core sees), as float32."""
    return decode(encode(x, fmt), fmt).astype(np.float32)


# ---- UE4M3 (NVFP4 block scale) ------------------------------------------------

def encode_ue4m3(x) -> np.ndarray:
    """Unsigned E4M3 of a non-negative fp32 value (RN-even, saturate at 448)."""
    x32 = np.asarray(x, dtype=np.float32)
    assert not np.any(np.signbit(x32) & (x32 != 0)), "UE4M3 input must be non-negative"
    return encode(np.abs(x32), "e4m3")


def decode_ue4m3(codes) -> np.ndarray:
    return decode(np.asarray(codes) & 0x7F, "e4m3")


# ---- E8M0 (MXFP8 block scale) -------------------------------------------------

def decode_e8m0(b) -> np.ndarray:
    b = np.asarray(b).astype(np.int64)
    v = np.exp2((b - 127).astype(np.float64))
    return np.where(b == 0xFF, np.nan, v)


def floor_log2(a) -> np.ndarray:
    """floor(log2(a)) for finite a > 0, exact (via frexp on the fp64 value)."""
    _, ex = np.frexp(np.asarray(a, dtype=np.float64))
    return ex.astype(np.int64) - 1


# ---- bf16 helpers (host representation: uint16 bit patterns) ------------------

def bf16_bits_to_f32(u16) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    u = np.asarray(u16).astype(np.uint32) << 16
    return u.view(np.float32)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 values to bf16 (RN-even via fp32 then bf16), as uint16 bits.

    Double rounding through fp32 only matters for values within 2**-24 relative
    of a bf16 midpoint; used for GEMM reference outputs only (tolerance checks).
    """
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r
