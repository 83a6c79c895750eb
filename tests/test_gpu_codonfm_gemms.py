"""Full-size parity of a layer's 12 GEMMs at the CodonFM-5B shapes, in every kind.

("How to Optimize Transformer-Based Models for Low-Precision Training", sections
"モデル設定とトレーニング入力" and "autocast モードの使用と事前量子化の比較": M = 31 x 512 =
15872 tokens, hidden 4096, intermediate 16384; QKV, attention output, MLP up and MLP down,
each as Fprop, Dgrad and Wgrad, benchmarked separately because their aspect ratios
differ.)

For each linear the inputs are drawn once (X ~ N(0, 1), W ~ N(0, 0.02^2), dY ~ N(0, 1e-3^2),
bias ~ N(0, 0.02^2), bf16).  Per pass and kind the library quantizes the two operands in
the orientation that GEMM consumes, as autocast does (FP8 CurrentScaling HYBRID; MXFP8; NVFP4
with 16 x 16 weight blocks, the random Hadamard transform on the Wgrad operands and
stochastic rounding of dY), then runs the GEMM to fp32 and to bf16 outputs.  The oracle
quantizes, on its own, the operand rows behind 64 sampled rows and 64 sampled columns of D
(with the whole tensors' amaxes -- for NVFP4's rotated copies the amax after the rotation),
takes their fp64 product and applies the GEMM bar: relative Frobenius error <= 1e-3 and an
element-wise bound (tests/gpu_util.check_gemm).
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from oracle import quantize as Q
from oracle import recipes as Rc
from synthetic import gaussian, rht_sign_mask, seed_for
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

M = 15872
LINEARS = [("qkv", 4096, 12288), ("attn_out", 4096, 4096), ("mlp_up", 4096, 16384), ("mlp_down", 16384, 4096)]
PASSES = ("fprop", "dgrad", "wgrad")
KINDS = ("bf16", "fp8", "mxfp8", "nvfp4")
NSAMPLE = 64
SIGNS = rht_sign_mask(41)
SR_SEED, SR_OFFSET = 9, 2
FP8_FMT = {"x": "e4m3", "w": "e4m3", "dy": "e5m2"}           # HYBRID
NV_FLAGS = {("x", "row"): 0, ("x", "col"): te.NVFP4_RHT_COL, ("w", "row"): te.NVFP4_2D,
            ("w", "col"): te.NVFP4_2D, ("dy", "row"): te.NVFP4_SR, ("dy", "col"): te.NVFP4_RHT_COL | te.NVFP4_SR}
# operands (tensor, copy) of each pass: A, B; D rows index A's copy rows, D columns B's
OPERANDS = {"fprop": (("x", "row"), ("w", "row")), "dgrad": (("dy", "row"), ("w", "col")),
            "wgrad": (("dy", "col"), ("x", "col"))}


class LinearData:
    """Host and device inputs of one linear, with the oracle's whole-tensor amaxes (cached)."""

    def __init__(self, idx: int):
        self.name, self.kin, self.nout = LINEARS[idx]
        s = [seed_for(7, idx, t) for t in range(4)]
        host = {"x": gaussian((M, self.kin), 1.0, s[0]), "w": gaussian((self.nout, self.kin), 0.02, s[1]),
                "dy": gaussian((M, self.nout), 1e-3, s[2])}
        self.bias = gaussian((self.nout,), 0.02, s[3], dtype=torch.float32)
        self.dev = {k: v.to(G.DEV) for k, v in host.items()}
        self.bias_dev = self.bias.to(G.DEV)
        self.f32 = {k: G.f32_np(v) for k, v in host.items()}
        self._amax, self._ramax = {}, {}

    def amax(self, t):
        if t not in self._amax:
            self._amax[t] = Q.amax(self.f32[t])
        return self._amax[t]

    def rot_amax(self, t):
        """Amax of the col copy after the 16-point rotation along the token dimension."""
        if t not in self._ramax:
            a = self.f32[t]
            self._ramax[t] = np.float32(max(float(Q.amax(Q.rht16(np.ascontiguousarray(a[:, c:c + 256].T), SIGNS)))
                                            for c in range(0, a.shape[1], 256)))
        return self._ramax[t]


_CACHE = {}


def _data(idx):
    if idx not in _CACHE:
        _CACHE.clear()
        torch.cuda.empty_cache()
        _CACHE[idx] = LinearData(idx)
    return _CACHE[idx]


# ---- the oracle's operand rows -----------------------------------------------------------------

def _copy_rows(t32, copy, idx):
    """Rows ``idx`` of the row copy (rows of t) or of the col copy (columns of t, as rows)."""
    return t32[idx] if copy == "row" else np.ascontiguousarray(t32[:, idx].T)


def oracle_operand(kind, d: LinearData, t, copy, idx):
    t32 = d.f32[t]
    if kind == "bf16":
        return _copy_rows(t32, copy, idx).astype(np.float64)
    if kind == "fp8":
        fmt = FP8_FMT[t]
        s, si = Rc.current_scale(d.amax(t), fmt)
        return Q.fp8_dequant(Q.fp8_cast(_copy_rows(t32, copy, idx), s, fmt), si, fmt)
    if kind == "mxfp8":
        return Q.mxfp8_dequant(*Q.mxfp8_quantize(_copy_rows(t32, copy, idx)))
    # NVFP4
    flags = NV_FLAGS[(t, copy)]
    src = t32 if copy == "row" else t32.T          # the copy's logical rows
    if flags & te.NVFP4_2D:
        out = []
        for r in idx:                              # the 16-row group holding r, 16 x 16 blocks
            g = int(r) - int(r) % 16
            grp = np.ascontiguousarray(src[g:g + 16])
            out.append(Q.nvfp4_dequant(*Q.nvfp4_quantize(grp, d.amax(t), block2d=True))[int(r) - g])
        return np.stack(out)
    rot = bool(flags & te.NVFP4_RHT_COL)
    amax = d.rot_amax(t) if rot else d.amax(t)
    out = []
    for r in idx:
        row = np.ascontiguousarray(src[int(r):int(r) + 1])
        if rot:
            row = Q.rht16(row, SIGNS)
        sr = (dict(seed=SR_SEED, copy_id=0 if copy == "row" else 1, offset=SR_OFFSET, row0=int(r),
                   cols=src.shape[1]) if flags & te.NVFP4_SR else None)
        out.append(Q.nvfp4_dequant(*Q.nvfp4_quantize(row, amax, sr=sr))[0])
    return np.stack(out)


# ---- the library's operands and GEMM --------------------------------------------------------------

def _quantize(kind, d: LinearData, t, copy):
    x = d.dev[t]
    R, C = x.shape
    row, col = copy == "row", copy == "col"
    if kind == "fp8":
        q = G.u8(R, C) if row else G.u8(C, R)
        amax, sinv = G.scalar(), G.scalar()
        te.te_quantize_fp8(x, te.E4M3 if FP8_FMT[t] == "e4m3" else te.E5M2, compute_scale=1,
                           q_row=q if row else None, q_col=q if col else None, amax_out=amax, scale_inv_out=sinv)
        return q, sinv
    if kind == "mxfp8":
        q = G.u8(R, C) if row else G.u8(C, R)
        s = G.u8(te.te_scale_bytes(te.E8M0, R, C) if row else te.te_scale_bytes(te.E8M0, C, R))
        te.te_quantize_mxfp8(x, q if row else None, s if row else None, q if col else None, s if col else None)
        return q, s
    flags = NV_FLAGS[(t, copy)]
    rot = bool(flags & te.NVFP4_RHT_COL)
    a, ar = G.scalar(), G.scalar()
    te.te_amax_reduce(x, None if rot else a, ar if rot else None, SIGNS)
    q = G.u8(R, C // 2) if row else G.u8(C, R // 2)
    s = G.u8(te.te_scale_bytes(te.UE4M3, R, C) if row else te.te_scale_bytes(te.UE4M3, C, R))
    g = G.scalar()
    none3 = (None, None, None)
    te.te_quantize_nvfp4(x, flags, SIGNS, SR_SEED, SR_OFFSET, a, ar, *((q, s, g) if row else none3),
                         *((q, s, g) if col else none3))
    return q, s, g


def _gemm(kind, d: LinearData, pass_, out_dtype):
    (ta, ca), (tb, cb) = OPERANDS[pass_]
    bias = d.bias_dev if pass_ == "fprop" else None
    rows_d = d.dev[ta].shape[0] if ca == "row" else d.dev[ta].shape[1]
    cols_d = d.dev[tb].shape[0] if cb == "row" else d.dev[tb].shape[1]
    D = torch.empty(rows_d, cols_d, dtype=out_dtype, device=G.DEV)
    if kind == "bf16":
        lay = {"row": te.K_MAJOR, "col": te.MN_MAJOR}
        te.te_gemm_bf16(d.dev[ta], d.dev[tb], D, bias, a_layout=lay[ca], b_layout=lay[cb])
        return D
    qa, qb = _quantize(kind, d, ta, ca), _quantize(kind, d, tb, cb)
    if kind == "fp8":
        fa = te.E4M3 if FP8_FMT[ta] == "e4m3" else te.E5M2
        fb = te.E4M3 if FP8_FMT[tb] == "e4m3" else te.E5M2
        te.te_gemm_fp8(qa[0], fa, qb[0], fb, qa[1], qb[1], D, bias)
    elif kind == "mxfp8":
        te.te_gemm_mxfp8(qa[0], qa[1], qb[0], qb[1], D, bias)
    else:
        te.te_gemm_nvfp4(qa[0], qa[1], qa[2], qb[0], qb[1], qb[2], D, bias)
    return D


CASES = [(li, p, k) for li in range(len(LINEARS)) for p in PASSES for k in KINDS]


@pytest.mark.parametrize("li,pass_,kind", CASES,
                         ids=[f"{LINEARS[li][0]}-{p}-{k}" for li, p, k in CASES])
def test_codonfm_gemm_full_size_sampled(li, pass_, kind):
    d = _data(li)
    (ta, ca), (tb, cb) = OPERANDS[pass_]
    rng = np.random.default_rng(1000 * li + 10 * PASSES.index(pass_) + KINDS.index(kind))
    for out_dtype in (torch.float32, torch.bfloat16):
        D = _gemm(kind, d, pass_, out_dtype)
        rows = np.sort(rng.choice(D.shape[0], NSAMPLE, replace=False))
        cols = np.sort(rng.choice(D.shape[1], NSAMPLE, replace=False))
        sub = D[torch.from_numpy(rows).to(G.DEV)][:, torch.from_numpy(cols).to(G.DEV)]
        torch.cuda.synchronize()
        G.check_no_device_error()
        got = G.f32_np(sub) if out_dtype == torch.bfloat16 else sub.cpu().numpy()
        a64 = oracle_operand(kind, d, ta, ca, rows)
        b64 = oracle_operand(kind, d, tb, cb, cols)
        bias = d.bias.numpy()[cols] if pass_ == "fprop" else None
        G.check_gemm(got, a64, b64, bias=bias, bf16_out=out_dtype == torch.bfloat16,
                     what=f"{d.name} {pass_} {kind} {out_dtype}")
        del D, sub
