"""GPU parity of the tcgen05 GEMMs against the oracle's fp64 products.

Both sides quantize the same seeded inputs independently (the quantizers are
bit-exact, pinned in test_gpu_quant); the oracle then multiplies its own
dequantized operands in fp64.  Bar: relative Frobenius error <= 1e-3, on fp32
outputs against the fp64 product and on bf16 outputs against the bf16-rounded
fp64 product.  Shapes cover all three passes of a linear layer with ragged
tiles; the CodonFM shapes (M = 15872) are checked on sampled sub-blocks.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from oracle import formats as F
from oracle import gemm as OG
from oracle import quantize as Q
from oracle import recipes as Rc
from synthetic import gaussian, rht_sign_mask
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
TOL = 1e-3


def _cmp(D, A64, B64, bias, what):
    """Parity of a whole output D against the oracle: rel-Frobenius and element-wise bar."""
    bf16 = D.dtype == torch.bfloat16
    got = G.f32_np(D) if bf16 else D.detach().cpu().numpy()
    return G.check_gemm(got, A64, B64, bias=bias, bf16_out=bf16, what=what)


def _linear(M, Kin, Nout, seed):
    x = gaussian((M, Kin), 1.0, seed)
    w = gaussian((Nout, Kin), 0.02, seed + 1)
    dy = gaussian((M, Nout), 1e-3, seed + 2)
    b = gaussian((Nout,), 0.02, seed + 3, dtype=torch.float32)
    return x.to(G.DEV), w.to(G.DEV), dy.to(G.DEV), b.to(G.DEV)


SMALL = [(272, 208, 528), (16, 32, 48), (1024, 768, 768), (384, 512, 256)]


# ---- BF16 ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("M,Kin,Nout", SMALL)
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_bf16_three_passes(M, Kin, Nout, out):
    x, w, dy, b = _linear(M, Kin, Nout, 100)
    x32, w32, dy32 = G.f32_np(x), G.f32_np(w), G.f32_np(dy)
    KM, MN = te.K_MAJOR, te.MN_MAJOR
    # dgrad reads W [Nout, Kin] as B stored [K, N]; wgrad reads dY and X as stored [K, M] / [K, N]
    passes = [("fprop", x, KM, w, KM, x32, w32, b, (M, Nout)), ("dgrad", dy, KM, w, MN, dy32, w32.T, None, (M, Kin)),
              ("wgrad", dy, MN, x, MN, dy32.T, x32.T, None, (Nout, Kin)),
              ("fprop-transposed-copies", x, KM, w.t().contiguous(), MN, x32, w32, b, (M, Nout))]
    for name, A, la, B, lb, A32, B32, bias, dshape in passes:
        D = torch.empty(*dshape, dtype=out, device=G.DEV)
        te.te_gemm_bf16(A, B, D, bias, a_layout=la, b_layout=lb)
        torch.cuda.synchronize()
        _cmp(D, A32, B32, None if bias is None else b.cpu().numpy(), f"bf16 {name}")
    G.check_no_device_error()


# ---- FP8 -----------------------------------------------------------------------------------------

def _fp8_current(t, fmt):
    code = te.E4M3 if fmt == "e4m3" else te.E5M2
    R, C = t.shape
    q_row, q_col = G.u8(R, C), G.u8(C, R)
    amax, sinv = G.scalar(), G.scalar()
    te.te_quantize_fp8(t, code, compute_scale=1, q_row=q_row, q_col=q_col, amax_out=amax, scale_inv_out=sinv)
    return q_row, q_col, sinv


def _fp8_oracle(t32, fmt):
    s, si = Rc.current_scale(Q.amax(t32), fmt)
    q_row, q_col, _, _ = Q.fp8_quantize(t32, s, fmt)
    return Q.fp8_dequant(q_row, si, fmt), Q.fp8_dequant(q_col, si, fmt)


@pytest.mark.parametrize("M,Kin,Nout", SMALL)
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_fp8_three_passes(M, Kin, Nout, out):
    x, w, dy, b = _linear(M, Kin, Nout, 200)
    xr, xc, xs = _fp8_current(x, "e4m3")
    wr, wc, ws = _fp8_current(w, "e4m3")
    dr, dc, ds = _fp8_current(dy, "e5m2")
    ox_r, ox_c = _fp8_oracle(G.f32_np(x), "e4m3")
    ow_r, ow_c = _fp8_oracle(G.f32_np(w), "e4m3")
    od_r, od_c = _fp8_oracle(G.f32_np(dy), "e5m2")
    E4, E5 = te.E4M3, te.E5M2
    passes = [("fprop", xr, E4, xs, wr, E4, ws, b, ox_r, ow_r),
              ("dgrad", dr, E5, ds, wc, E4, ws, None, od_r, ow_c),
              ("wgrad", dc, E5, ds, xc, E4, xs, None, od_c, ox_c)]
    for name, A, fa, sa, B, fb, sb, bias, A64, B64 in passes:
        D = torch.empty(A.shape[0], B.shape[0], dtype=out, device=G.DEV)
        te.te_gemm_fp8(A, fa, B, fb, sa, sb, D, bias)
        torch.cuda.synchronize()
        _cmp(D, A64, B64, None if bias is None else b.cpu().numpy(), f"fp8 {name}")
    G.check_no_device_error()


def test_fp8_small_integers_exact():
    M, N, K = 256, 512, 384
    rng = np.random.default_rng(3)
    ai = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    bi = rng.integers(-8, 9, size=(N, K)).astype(np.float32)
    A = torch.from_numpy(ai).to(G.DEV)
    B = torch.from_numpy(bi).to(G.DEV)
    qa, qb = G.u8(M, K), G.u8(N, K)
    sa, sb = G.scalar(4.0), G.scalar(0.5)
    ia, ib = G.scalar(), G.scalar()
    te.te_quantize_fp8(A, te.E4M3, scale=sa, q_row=qa, scale_inv_out=ia)
    te.te_quantize_fp8(B, te.E4M3, scale=sb, q_row=qb, scale_inv_out=ib)
    D = torch.empty(M, N, dtype=torch.float32, device=G.DEV)
    te.te_gemm_fp8(qa, te.E4M3, qb, te.E4M3, ia, ib, D)
    torch.cuda.synchronize()
    exact = (ai.astype(np.int64) @ bi.astype(np.int64).T).astype(np.float32)
    np.testing.assert_array_equal(D.cpu().numpy(), exact)


# ---- MXFP8 ---------------------------------------------------------------------------------------

def _mx(t):
    R, C = t.shape
    q_row, q_col = G.u8(R, C), G.u8(C, R)
    s_row = G.u8(te.te_scale_bytes(te.E8M0, R, C))
    s_col = G.u8(te.te_scale_bytes(te.E8M0, C, R))
    te.te_quantize_mxfp8(t, q_row, s_row, q_col, s_col)
    return q_row, s_row, q_col, s_col


def _mx_oracle(t32):
    qr, sr = Q.mxfp8_quantize(t32)
    qc, sc = Q.mxfp8_quantize(np.ascontiguousarray(t32.T))
    return Q.mxfp8_dequant(qr, sr), Q.mxfp8_dequant(qc, sc)


MX_SMALL = [(288, 224, 544), (32, 64, 96), (1024, 768, 768)]


@pytest.mark.parametrize("M,Kin,Nout", MX_SMALL)
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_mxfp8_three_passes(M, Kin, Nout, out):
    x, w, dy, b = _linear(M, Kin, Nout, 300)
    xr, xsr, xc, xsc = _mx(x)
    wr, wsr, wc, wsc = _mx(w)
    dr, dsr, dc, dsc = _mx(dy)
    ox_r, ox_c = _mx_oracle(G.f32_np(x))
    ow_r, ow_c = _mx_oracle(G.f32_np(w))
    od_r, od_c = _mx_oracle(G.f32_np(dy))
    passes = [("fprop", xr, xsr, wr, wsr, b, ox_r, ow_r), ("dgrad", dr, dsr, wc, wsc, None, od_r, ow_c),
              ("wgrad", dc, dsc, xc, xsc, None, od_c, ox_c)]
    for name, A, sA, B, sB, bias, A64, B64 in passes:
        D = torch.empty(A.shape[0], B.shape[0], dtype=out, device=G.DEV)
        te.te_gemm_mxfp8(A, sA, B, sB, D, bias)
        torch.cuda.synchronize()
        _cmp(D, A64, B64, None if bias is None else b.cpu().numpy(), f"mxfp8 {name}")
    G.check_no_device_error()


# ---- NVFP4 ---------------------------------------------------------------------------------------

SIGNS = rht_sign_mask(41)


def _nv(t, flags, seed=0, offset=0):
    R, C = t.shape
    a, ar = G.scalar(), G.scalar()
    te.te_amax_reduce(t, a, ar, SIGNS)
    q_row, q_col = G.u8(R, C // 2), G.u8(C, R // 2)
    s_row, s_col = G.u8(te.te_scale_bytes(te.UE4M3, R, C)), G.u8(te.te_scale_bytes(te.UE4M3, C, R))
    g_row, g_col = G.scalar(), G.scalar()
    te.te_quantize_nvfp4(t, flags, SIGNS, seed, offset, a, ar, q_row, s_row, g_row, q_col, s_col, g_col)
    return q_row, s_row, g_row, q_col, s_col, g_col


def _nv_oracle(t32, flags, seed=0, offset=0):
    R, C = t32.shape
    sr = bool(flags & te.NVFP4_SR)
    two_d = bool(flags & te.NVFP4_2D)
    A = Q.amax(t32)
    q, s, d = Q.nvfp4_quantize(t32, A, block2d=two_d,
                               sr=dict(seed=seed, copy_id=0, offset=offset, row0=0, cols=C) if sr else None)
    row = Q.nvfp4_dequant(q, s, d)
    z = np.ascontiguousarray(t32.T)
    if flags & te.NVFP4_RHT_COL:
        z = Q.rht16(z, SIGNS)
    q, s, d = Q.nvfp4_quantize(z, Q.amax(z), block2d=two_d,
                               sr=dict(seed=seed, copy_id=1, offset=offset, row0=0, cols=R) if sr else None)
    return row, Q.nvfp4_dequant(q, s, d)


NV_SMALL = [(288, 224, 544), (32, 64, 96), (1024, 768, 768)]
X_FLAGS = te.NVFP4_RHT_COL
W_FLAGS = te.NVFP4_2D
DY_FLAGS = te.NVFP4_RHT_COL | te.NVFP4_SR


@pytest.mark.parametrize("M,Kin,Nout", NV_SMALL)
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_nvfp4_three_passes(M, Kin, Nout, out):
    x, w, dy, b = _linear(M, Kin, Nout, 400)
    xq = _nv(x, X_FLAGS)
    wq = _nv(w, W_FLAGS)
    dq = _nv(dy, DY_FLAGS, seed=5, offset=1)
    ox_r, ox_c = _nv_oracle(G.f32_np(x), X_FLAGS)
    ow_r, ow_c = _nv_oracle(G.f32_np(w), W_FLAGS)
    od_r, od_c = _nv_oracle(G.f32_np(dy), DY_FLAGS, seed=5, offset=1)
    passes = [("fprop", xq[0:3], wq[0:3], b, ox_r, ow_r), ("dgrad", dq[0:3], wq[3:6], None, od_r, ow_c),
              ("wgrad", dq[3:6], xq[3:6], None, od_c, ox_c)]
    for name, (A, sA, gA), (B, sB, gB), bias, A64, B64 in passes:
        D = torch.empty(A.shape[0], B.shape[0], dtype=out, device=G.DEV)
        te.te_gemm_nvfp4(A, sA, gA, B, sB, gB, D, bias)
        torch.cuda.synchronize()
        _cmp(D, A64, B64, None if bias is None else b.cpu().numpy(), f"nvfp4 {name}")
    G.check_no_device_error()


# ---- CodonFM shapes, sampled sub-blocks -----------------------------------------------------------

def _sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, k, replace=False))


@pytest.mark.parametrize("kind", ["bf16", "fp8", "mxfp8", "nvfp4"])
def test_codonfm_attn_out_fprop_sampled(kind):
    M, K, N = 15872, 4096, 4096
    x = gaussian((M, K), 1.0, 501).to(G.DEV)
    w = gaussian((N, K), 0.02, 502).to(G.DEV)
    rows, cols = _sample(M, 128, 1), _sample(N, 128, 2)
    x32, w32 = G.f32_np(x), G.f32_np(w)
    D = torch.empty(M, N, dtype=torch.float32, device=G.DEV)
    if kind == "bf16":
        te.te_gemm_bf16(x, w, D)
        A64, B64 = x32[rows], w32[cols]
    elif kind == "fp8":
        xr, _, xs = _fp8_current(x, "e4m3")
        wr, _, ws = _fp8_current(w, "e4m3")
        te.te_gemm_fp8(xr, te.E4M3, wr, te.E4M3, xs, ws, D)
        sx, six = Rc.current_scale(Q.amax(x32), "e4m3")
        sw, siw = Rc.current_scale(Q.amax(w32), "e4m3")
        A64 = Q.fp8_dequant(Q.fp8_cast(x32[rows], sx, "e4m3"), six, "e4m3")
        B64 = Q.fp8_dequant(Q.fp8_cast(w32[cols], sw, "e4m3"), siw, "e4m3")
    elif kind == "mxfp8":
        xr, xsr, _, _ = _mx(x)
        wr, wsr, _, _ = _mx(w)
        te.te_gemm_mxfp8(xr, xsr, wr, wsr, D)
        A64 = Q.mxfp8_dequant(*Q.mxfp8_quantize(x32[rows]))
        B64 = Q.mxfp8_dequant(*Q.mxfp8_quantize(w32[cols]))
    else:
        xq = _nv(x, 0)
        wq = _nv(w, W_FLAGS)
        te.te_gemm_nvfp4(xq[0], xq[1], xq[2], wq[0], wq[1], wq[2], D)
        A64 = Q.nvfp4_dequant(*Q.nvfp4_quantize(x32[rows], Q.amax(x32)))
        g16 = (cols // 16) * 16
        blocks = np.unique(g16)
        wsub = np.concatenate([w32[bb:bb + 16] for bb in blocks])                 # whole 16-row groups for 2D
        wq_o = Q.nvfp4_dequant(*Q.nvfp4_quantize(wsub, Q.amax(w32), block2d=True))
        idx = {int(bb): i for i, bb in enumerate(blocks)}
        B64 = np.stack([wq_o[idx[int(c - c % 16)] * 16 + c % 16] for c in cols])
    torch.cuda.synchronize()
    got = D.cpu().numpy()[np.ix_(rows, cols)]
    G.check_gemm(got, A64, B64, what=kind)
    G.check_no_device_error()


@pytest.mark.parametrize("kind", ["bf16", "fp8"])
def test_codonfm_mlp_down_fprop_sampled(kind):
    """The longest contraction of the layer: 15872 x 4096 x 16384 (MLP down, Fprop)."""
    M, K, N = 15872, 16384, 4096
    x = gaussian((M, K), 1.0, 801).to(G.DEV)
    w = gaussian((N, K), 0.02, 802).to(G.DEV)
    b = gaussian((N,), 0.02, 803, dtype=torch.float32).to(G.DEV)
    rows, cols = _sample(M, 96, 5), _sample(N, 96, 6)
    x32, w32 = G.f32_np(x), G.f32_np(w)
    D = torch.empty(M, N, dtype=torch.bfloat16, device=G.DEV)
    if kind == "bf16":
        te.te_gemm_bf16(x, w, D, b)
        A64, B64 = x32[rows], w32[cols]
    else:
        xr, _, xs = _fp8_current(x, "e4m3")
        wr, _, ws = _fp8_current(w, "e4m3")
        te.te_gemm_fp8(xr, te.E4M3, wr, te.E4M3, xs, ws, D, b)
        sx, six = Rc.current_scale(Q.amax(x32), "e4m3")
        sw, siw = Rc.current_scale(Q.amax(w32), "e4m3")
        A64 = Q.fp8_dequant(Q.fp8_cast(x32[rows], sx, "e4m3"), six, "e4m3")
        B64 = Q.fp8_dequant(Q.fp8_cast(w32[cols], sw, "e4m3"), siw, "e4m3")
    torch.cuda.synchronize()
    got = G.f32_np(D)[np.ix_(rows, cols)]
    G.check_gemm(got, A64, B64, bias=b.cpu().numpy()[cols], bf16_out=True, what=kind)
    G.check_no_device_error()


@pytest.mark.parametrize("kind", ["fp8", "nvfp4"])
def test_codonfm_wgrad_sampled(kind):
    """dW = dY^T X for attention output: 4096 x 4096 x 15872 (contraction over tokens)."""
    M, H = 15872, 4096
    x = gaussian((M, H), 1.0, 601).to(G.DEV)
    dy = gaussian((M, H), 1e-3, 602).to(G.DEV)
    rows, cols = _sample(H, 96, 3), _sample(H, 96, 4)
    x32, dy32 = G.f32_np(x), G.f32_np(dy)
    D = torch.empty(H, H, dtype=torch.float32, device=G.DEV)
    if kind == "fp8":
        _, xc, xs = _fp8_current(x, "e4m3")
        _, dc, ds = _fp8_current(dy, "e5m2")
        te.te_gemm_fp8(dc, te.E5M2, xc, te.E4M3, ds, xs, D)
        sx, six = Rc.current_scale(Q.amax(x32), "e4m3")
        sd, sid = Rc.current_scale(Q.amax(dy32), "e5m2")
        A64 = Q.fp8_dequant(Q.fp8_cast(np.ascontiguousarray(dy32[:, rows].T), sd, "e5m2"), sid, "e5m2")
        B64 = Q.fp8_dequant(Q.fp8_cast(np.ascontiguousarray(x32[:, cols].T), sx, "e4m3"), six, "e4m3")
    else:
        xq = _nv(x, X_FLAGS)
        dq = _nv(dy, DY_FLAGS, seed=9, offset=2)
        te.te_gemm_nvfp4(dq[3], dq[4], dq[5], xq[3], xq[4], xq[5], D)

        def rot_amax(t32):
            return np.float32(max(float(Q.amax(Q.rht16(np.ascontiguousarray(t32[:, c:c + 512].T), SIGNS)))
                                  for c in range(0, t32.shape[1], 512)))
        Ad, Ax = rot_amax(dy32), rot_amax(x32)
        A64 = np.concatenate([Q.nvfp4_dequant(*Q.nvfp4_quantize(
            Q.rht16(np.ascontiguousarray(dy32[:, r:r + 1].T), SIGNS), Ad,
            sr=dict(seed=9, copy_id=1, offset=2, row0=int(r), cols=M))) for r in rows])
        B64 = np.concatenate([Q.nvfp4_dequant(*Q.nvfp4_quantize(
            Q.rht16(np.ascontiguousarray(x32[:, c:c + 1].T), SIGNS), Ax)) for c in cols])
    torch.cuda.synchronize()
    got = D.cpu().numpy()[np.ix_(rows, cols)]
    G.check_gemm(got, A64, B64, what=kind)
    G.check_no_device_error()


def test_gemm_rejects_bad_shapes():
    A = torch.zeros(32, 40, dtype=torch.bfloat16, device=G.DEV)
    D = torch.empty(32, 32, dtype=torch.float32, device=G.DEV)
    with pytest.raises(te.TEError) as ei:
        te.te_gemm_bf16(A, torch.zeros(32, 40, dtype=torch.bfloat16, device=G.DEV), D)   # K = 40
    assert ei.value.status == 2


# ---- Wgrad accumulated into an fp32 main gradient -----------------------------------------------

@pytest.mark.parametrize("kind", ["bf16", "fp8", "mxfp8", "nvfp4"])
def test_wgrad_accumulates_into_fp32_main_grad(kind):
    # two micro-batches of tokens; dW of each is added into one fp32 buffer that already
    # holds a gradient, in place (accumulate=1): D = D0 + dW_1 + dW_2
    M, Kin, Nout = 256, 288, 224
    rng = np.random.default_rng(17)
    d0 = (rng.standard_normal((Nout, Kin)) * 0.01).astype(np.float32)
    D = torch.from_numpy(d0.copy()).to(G.DEV)
    ref = d0.astype(np.float64)
    for mb in range(2):
        x, w, dy, b = _linear(M, Kin, Nout, 700 + 10 * mb)
        x32, dy32 = G.f32_np(x), G.f32_np(dy)
        if kind == "bf16":
            te.te_gemm_bf16(dy, x, D, None, a_layout=te.MN_MAJOR, b_layout=te.MN_MAJOR, accumulate=1)
            A64, B64 = dy32.T, x32.T
        elif kind == "fp8":
            _, dc, ds = _fp8_current(dy, "e5m2")
            _, xc, xs = _fp8_current(x, "e4m3")
            te.te_gemm_fp8(dc, te.E5M2, xc, te.E4M3, ds, xs, D, accumulate=1)
            A64, B64 = _fp8_oracle(dy32, "e5m2")[1], _fp8_oracle(x32, "e4m3")[1]
        elif kind == "mxfp8":
            _, _, dc, dsc = _mx(dy)
            _, _, xc, xsc = _mx(x)
            te.te_gemm_mxfp8(dc, dsc, xc, xsc, D, accumulate=1)
            A64, B64 = _mx_oracle(dy32)[1], _mx_oracle(x32)[1]
        else:
            dq = _nv(dy, te.NVFP4_RHT_COL)
            xq = _nv(x, te.NVFP4_RHT_COL)
            te.te_gemm_nvfp4(dq[3], dq[4], dq[5], xq[3], xq[4], xq[5], D, accumulate=1)
            A64 = _nv_oracle(dy32, te.NVFP4_RHT_COL)[1]
            B64 = _nv_oracle(x32, te.NVFP4_RHT_COL)[1]
        torch.cuda.synchronize()
        ref = OG.gemm_accumulate(ref, A64, B64)
    got = D.cpu().numpy().astype(np.float64)
    # the bar applies to the accumulated increment (the product); D0 itself must survive
    err = OG.rel_frobenius(got - d0, ref - d0)
    assert err <= TOL, f"{kind} wgrad accumulate: rel-Frobenius {err:.3e}"
    G.check_no_device_error()


def test_accumulate_of_zero_product_keeps_main_grad_bits():
    M, N, K = 256, 256, 128
    d0 = np.random.default_rng(2).standard_normal((M, N)).astype(np.float32)
    D = torch.from_numpy(d0.copy()).to(G.DEV)
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=G.DEV)
    B = torch.zeros(N, K, dtype=torch.bfloat16, device=G.DEV)
    te.te_gemm_bf16(A, B, D, None, accumulate=1)
    te.te_gemm_bf16(A, B, D, None, accumulate=1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(D.cpu().numpy().view(np.uint32), d0.view(np.uint32))
    with pytest.raises(te.TEError):
        te.te_gemm_bf16(A, B, torch.empty(M, N, dtype=torch.bfloat16, device=G.DEV), None, accumulate=1)


@pytest.mark.parametrize("kind", ["bf16", "fp8", "mxfp8", "nvfp4"])
def test_several_tiles_per_pair_ragged_k(kind):
    """2304 x 4352 outputs are 153 tiles, three per CTA pair, so the pairs' second tiles walk K
    backwards; K = 1056 leaves the last 128-byte k-tile partly outside the operands (zero-filled
    by TMA) on every kind.  The whole output against the oracle's fp64 product."""
    M, N, K = 2304, 4352, 1056
    x = gaussian((M, K), 1.0, 611).to(G.DEV)
    w = gaussian((N, K), 0.02, 612).to(G.DEV)
    b = gaussian((N,), 0.02, 613, dtype=torch.float32).to(G.DEV)
    x32, w32 = G.f32_np(x), G.f32_np(w)
    D = torch.empty(M, N, dtype=torch.bfloat16, device=G.DEV)
    if kind == "bf16":
        te.te_gemm_bf16(x, w, D, b)
        A64, B64 = x32, w32
    elif kind == "fp8":
        xr, _, xs = _fp8_current(x, "e4m3")
        wr, _, ws = _fp8_current(w, "e4m3")
        te.te_gemm_fp8(xr, te.E4M3, wr, te.E4M3, xs, ws, D, b)
        A64, B64 = _fp8_oracle(x32, "e4m3")[0], _fp8_oracle(w32, "e4m3")[0]
    elif kind == "mxfp8":
        xr, xsr, _, _ = _mx(x)
        wr, wsr, _, _ = _mx(w)
        te.te_gemm_mxfp8(xr, xsr, wr, wsr, D, b)
        A64 = Q.mxfp8_dequant(*Q.mxfp8_quantize(x32))
        B64 = Q.mxfp8_dequant(*Q.mxfp8_quantize(w32))
    else:
        xq, wq = _nv(x, 0), _nv(w, W_FLAGS)
        te.te_gemm_nvfp4(xq[0], xq[1], xq[2], wq[0], wq[1], wq[2], D, b)
        A64 = Q.nvfp4_dequant(*Q.nvfp4_quantize(x32, Q.amax(x32)))
        B64 = Q.nvfp4_dequant(*Q.nvfp4_quantize(w32, Q.amax(w32), block2d=True))
    torch.cuda.synchronize()
    _cmp(D, A64, B64, b.cpu().numpy(), f"{kind} {M}x{N}x{K}")
    G.check_no_device_error()
