"""GPU parity of the quantizer kernels against the CPU oracle (bit-exact).

Shapes span several 64 x 64 tiles with a ragged tail; the CodonFM-sized case
(15872 x 4096, the QKV / attention-output / MLP-up input) is compared on
sampled rows of both copies, with the tensor-wide amax exact.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from oracle import formats as F
from oracle import quantize as Q
from oracle import recipes as Rc
from synthetic import gaussian, student_t_outliers, uniform, rht_sign_mask
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

RAGGED = [(272, 208), (16, 48), (1024, 768), (80, 1040)]


def _x(shape, dtype, seed, kind="gauss"):
    if kind == "uniform":
        t = uniform(shape, seed, dtype=dtype)
    elif kind == "t":
        t = student_t_outliers(shape, seed, dtype=dtype)
    else:
        t = gaussian(shape, 1.0, seed, dtype=dtype)
    return t.to(G.DEV)


# ---- amax --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_amax_and_rht_amax(shape, dtype):
    x = _x(shape, dtype, 11, "t")
    signs = rht_sign_mask(5)
    a, ar = G.amax(x, signs)
    x32 = G.f32_np(x)
    assert a == Q.amax(x32)
    assert ar == Q.amax(Q.rht16(np.ascontiguousarray(x32.T), signs))
    a2, _ = G.amax(x)
    assert a2 == a
    # the rotated amax alone (plain amax pointer NULL)
    ar_only = G.scalar(-1.0)
    te.te_amax_reduce(x, None, ar_only, signs)
    torch.cuda.synchronize()
    assert np.float32(ar_only.item()) == ar
    G.check_no_device_error()


def test_amax_empty_and_zero():
    x = torch.zeros(0, 32, dtype=torch.bfloat16, device=G.DEV)
    assert G.amax(x, 3) == (0.0, 0.0)
    z = torch.zeros(64, 64, dtype=torch.float32, device=G.DEV)
    z[5, 7] = -0.0
    assert G.amax(z, 3) == (0.0, 0.0)


def test_amax_full_size():
    x = gaussian((15872, 4096), 1.0, 77).to(G.DEV)
    signs = rht_sign_mask(9)
    a, ar = G.amax(x, signs)
    x32 = G.f32_np(x)
    assert a == Q.amax(x32)
    # exact over the whole tensor, in column slabs to bound host memory
    ref = max(float(Q.amax(Q.rht16(np.ascontiguousarray(x32[:, c:c + 512].T), signs))) for c in range(0, 4096, 512))
    assert float(ar) == ref


# ---- scale update -----------------------------------------------------------------------------------

@pytest.mark.parametrize("L,algo,margin,interval,bwd", [(16, 0, 0, 1, 0), (4, 1, 0, 1, 1), (4, 0, 1, 2, 0),
                                                         (1024, 0, 0, 1, 1), (1, 1, 3, 1, 0)])
def test_scale_update_matches_oracle(L, algo, margin, interval, bwd):
    n, steps = 37, 24
    rng = np.random.default_rng(L + algo)
    amaxes = (rng.standard_exponential((steps, n)) * np.exp2(rng.integers(-20, 20, size=(steps, n)))).astype(np.float32)
    amaxes[3, :5] = 0.0
    amaxes[6, 7] = np.inf
    amaxes[9, 11] = np.nan          # a NaN amax holds the scale while it is in the window (like Inf)
    recipe = te.te_recipe(te.E4M3, te.E5M2, L, algo, margin, interval)
    hist = torch.zeros(n * L, dtype=torch.float32, device=G.DEV)
    scale = torch.ones(n, dtype=torch.float32, device=G.DEV)
    sinv = torch.ones(n, dtype=torch.float32, device=G.DEV)
    fmt = "e5m2" if bwd else "e4m3"
    states = [Rc.DelayedScalingState(fmt, L, algo, margin, interval) for _ in range(n)]
    for t in range(steps):
        a = torch.from_numpy(amaxes[t]).to(G.DEV)
        te.te_scale_update(recipe, bwd, hist, a, scale, sinv, t)
        for i, st in enumerate(states):
            st.update(amaxes[t, i], t)
        torch.cuda.synchronize()
        G.assert_equal_codes(scale.cpu().numpy().view(np.uint32), np.array([s.scale for s in states], np.float32).view(np.uint32), f"scale step {t}")
        G.assert_equal_codes(sinv.cpu().numpy().view(np.uint32), np.array([s.scale_inv for s in states], np.float32).view(np.uint32), f"scale_inv step {t}")
    G.assert_equal_codes(hist.cpu().numpy().reshape(n, L).view(np.uint32), np.stack([s.hist for s in states]).view(np.uint32), "history")
    G.check_no_device_error()


# ---- FP8 -------------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_delayed_and_current(shape, dtype, fmt):
    code = te.E4M3 if fmt == "e4m3" else te.E5M2
    x = _x(shape, dtype, 21, "t")
    x32 = G.f32_np(x)
    # Delayed: an arbitrary prior scale (saturates part of the tensor)
    s = np.float32(F.FMAX[fmt] / 3.0)
    q_row, q_col, amax, sinv = G.fp8(x, code, scale=s)
    e_row, e_col, e_amax, e_sinv = Q.fp8_quantize(x32, s, fmt)
    G.assert_equal_codes(q_row, e_row, "delayed row")
    G.assert_equal_codes(q_col, e_col, "delayed col")
    assert amax == e_amax and sinv == e_sinv
    # Current: scale from the tensor's own amax
    q_row, q_col, amax, sinv = G.fp8(x, code, current=True)
    cs, csi = Rc.current_scale(Q.amax(x32), fmt)
    e_row, e_col, _, _ = Q.fp8_quantize(x32, cs, fmt)
    G.assert_equal_codes(q_row, e_row, "current row")
    G.assert_equal_codes(q_col, e_col, "current col")
    assert amax == Q.amax(x32) and sinv == csi
    G.check_no_device_error()


def test_fp8_encoder_structured_values():
    """Every distinct rounding decision of E4M3 / E5M2 (fp32 input, scale 1)."""
    s = np.arange(2, dtype=np.uint32)[:, None, None]
    e = np.arange(255, dtype=np.uint32)[None, :, None]            # finite exponents (+ inf handled below)
    m = np.arange(4096, dtype=np.uint32)[None, None, :]
    bits = ((s << 31) | (e << 23) | (m << 11)).reshape(-1)
    low = np.array([0, 1, 0x2AA, 0x7FF], dtype=np.uint32)
    allbits = (bits[:, None] | low[None, :]).reshape(-1)
    vals = np.concatenate([allbits.view(np.float32), np.array([np.inf, -np.inf] * 32, np.float32)])
    vals = vals[: (vals.size // 1024) * 1024].reshape(-1, 64)     # rows a multiple of 16
    x = torch.from_numpy(vals.copy()).to(G.DEV)
    for fmt, code in [("e4m3", te.E4M3), ("e5m2", te.E5M2)]:
        q_row, _, _, _ = G.fp8(x, code, scale=1.0, col=False)
        G.assert_equal_codes(q_row, F.encode(vals, fmt), fmt)


def test_fp8_full_size_sampled():
    x = gaussian((15872, 4096), 1.0, 31).to(G.DEV)
    q_row, q_col, amax, sinv = G.fp8(x, te.E4M3, current=True)
    x32 = G.f32_np(x)
    cs, csi = Rc.current_scale(Q.amax(x32), "e4m3")
    assert amax == Q.amax(x32) and sinv == csi
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(15872, 96, replace=False))
    cols = np.sort(rng.choice(4096, 96, replace=False))
    G.assert_equal_codes(q_row[rows], Q.fp8_cast(x32[rows], cs, "e4m3"), "row sample")
    G.assert_equal_codes(q_col[cols], Q.fp8_cast(np.ascontiguousarray(x32[:, cols].T), cs, "e4m3"), "col sample")


def test_nvfp4_rejects_non_32_dims():
    x = torch.zeros(48, 64, dtype=torch.bfloat16, device=G.DEV)
    with pytest.raises(te.TEError) as ei:
        G.nvfp4(x, 0, row=False, col=True)     # col copy contracts over 48 rows
    assert ei.value.status == 2


def test_fp8_rejects_bad_shapes():
    x = torch.zeros(24, 32, dtype=torch.bfloat16, device=G.DEV)
    with pytest.raises(te.TEError) as ei:
        G.fp8(x, te.E4M3, scale=1.0)
    assert ei.value.status == 2


# ---- MXFP8 ---------------------------------------------------------------------------------------------

MX_SHAPES = [(96, 160), (1024, 768), (32, 32), (288, 224)]


@pytest.mark.parametrize("shape", MX_SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mxfp8_matches_oracle(shape, dtype):
    x = _x(shape, dtype, 41, "t")
    x32 = G.f32_np(x)
    x32[0, :32] = 0.0                         # a zero block
    x = torch.from_numpy(x32).to(dtype).to(G.DEV)
    x32 = G.f32_np(x)
    out = G.mxfp8(x)
    eq, es = Q.mxfp8_quantize(x32)
    G.assert_equal_codes(out["q_row"], eq, "row codes")
    G.assert_equal_codes(out["s_row"], es, "row scales")
    eq, es = Q.mxfp8_quantize(np.ascontiguousarray(x32.T))
    G.assert_equal_codes(out["q_col"], eq, "col codes")
    G.assert_equal_codes(out["s_col"], es, "col scales")
    # padding of the scale tensors is zero
    R, C = shape
    for raw, rows, cols in [(out["s_row_raw"], R, C), (out["s_col_raw"], C, R)]:
        logical_bytes = rows * (cols // 32)
        assert int(np.count_nonzero(raw)) <= logical_bytes
        assert raw.size == te.te_scale_bytes(te.E8M0, rows, cols)
    G.check_no_device_error()


def test_mxfp8_full_size_sampled():
    x = student_t_outliers((15872, 4096), 51).to(G.DEV)
    out = G.mxfp8(x)
    x32 = G.f32_np(x)
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(15872, 64, replace=False))
    cols = np.sort(rng.choice(4096, 64, replace=False))
    eq, es = Q.mxfp8_quantize(x32[rows])
    G.assert_equal_codes(out["q_row"][rows], eq, "row codes")
    G.assert_equal_codes(out["s_row"][rows], es, "row scales")
    eq, es = Q.mxfp8_quantize(np.ascontiguousarray(x32[:, cols].T))
    G.assert_equal_codes(out["q_col"][cols], eq, "col codes")
    G.assert_equal_codes(out["s_col"][cols], es, "col scales")


# ---- NVFP4 ---------------------------------------------------------------------------------------------

NV_SHAPES = [(64, 96), (1024, 768), (288, 224), (32, 32)]


def _nv_expect(x32, flags, signs, seed, offset):
    R, C = x32.shape
    A = Q.amax(x32)
    two_d = bool(flags & te.NVFP4_2D)
    sr = bool(flags & te.NVFP4_SR)
    row = Q.nvfp4_quantize(x32, A, block2d=two_d,
                           sr=dict(seed=seed, copy_id=0, offset=offset, row0=0, cols=C) if sr else None)
    zc = np.ascontiguousarray(x32.T)
    if flags & te.NVFP4_RHT_COL:
        zc = Q.rht16(zc, signs)
        Ac = Q.amax(zc)
    else:
        Ac = A
    col = Q.nvfp4_quantize(zc, Ac, block2d=two_d,
                           sr=dict(seed=seed, copy_id=1, offset=offset, row0=0, cols=R) if sr else None)
    return row, col


@pytest.mark.parametrize("shape", NV_SHAPES)
@pytest.mark.parametrize("flags", [0, 1, 2, 4, 6])   # plain, 2D (weights), RHT col, SR, RHT + SR (gradients)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_nvfp4_matches_oracle(shape, flags, dtype):
    x = _x(shape, dtype, 61 + flags, "t")
    signs = rht_sign_mask(17)
    seed, offset = 0x1234_5678_9ABCDEF, 3
    out = G.nvfp4(x, flags, signs, seed, offset)
    x32 = G.f32_np(x)
    (rq, rs, rd), (cq, cs, cd) = _nv_expect(x32, flags, signs, seed, offset)
    G.assert_equal_codes(out["q_row"], rq, "row codes")
    G.assert_equal_codes(out["s_row"], rs, "row scales")
    assert out["g_row"] == rd
    G.assert_equal_codes(out["q_col"], cq, "col codes")
    G.assert_equal_codes(out["s_col"], cs, "col scales")
    assert out["g_col"] == cd
    if flags & te.NVFP4_2D:
        G.assert_equal_codes(out["q_col"], out["q_row"].T, "2D transpose consistency")
    G.check_no_device_error()


def test_nvfp4_e2m1_encoder_structured_values():
    """Each 16-block holds a 6.0 so that S_enc = 448 and r = 1: q = E2M1(x) directly."""
    s = np.arange(2, dtype=np.uint32)[:, None, None]
    e = np.arange(120, 130, dtype=np.uint32)[None, :, None]       # magnitudes 2^-7 .. 2^2 (plus rounding up to 6)
    m = np.arange(4096, dtype=np.uint32)[None, None, :]
    bits = ((s << 31) | (e << 23) | (m << 11)).reshape(-1)
    low = np.array([0, 1, 0x7FF], dtype=np.uint32)
    vals = (bits[:, None] | low[None, :]).reshape(-1).view(np.float32)
    vals = np.concatenate([vals, np.array([5.0, 5.5, 6.0, 7.0, -5.0, -0.0, 0.25, 0.75], np.float32)])
    vals = np.clip(vals, -6.0, 6.0)
    nb = (vals.size // 15 // 128) * 128                    # whole [32 x 64] tiles of blocks
    blocks = vals[: nb * 15].reshape(nb, 15)
    blocks = np.concatenate([np.full((nb, 1), 6.0, np.float32), blocks], axis=1)
    z = blocks.reshape(nb // 4, 64)
    x = torch.from_numpy(np.ascontiguousarray(z)).to(G.DEV)
    out = G.nvfp4(x, 0, col=False)
    assert out["amax"] == 6.0
    G.assert_equal_codes(out["q_row"], F.encode(z, "e2m1"), "e2m1 encode")
    assert np.all(out["s_row"] == 0x7E)


def test_nvfp4_full_size_sampled():
    R, C = 15872, 4096
    dy = gaussian((R, C), 1e-3, 71).to(G.DEV)
    signs = rht_sign_mask(23)
    flags = te.NVFP4_RHT_COL | te.NVFP4_SR
    seed, offset = 99, 7
    out = G.nvfp4(dy, flags, signs, seed, offset)
    x32 = G.f32_np(dy)
    A = Q.amax(x32)
    assert out["amax"] == A
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(R, 32, replace=False))
    for r in rows:
        q, s, d = Q.nvfp4_quantize(x32[r:r + 1], A, sr=dict(seed=seed, copy_id=0, offset=offset, row0=int(r), cols=C))
        G.assert_equal_codes(out["q_row"][r:r + 1], q, f"row {r}")
        G.assert_equal_codes(out["s_row"][r:r + 1], s, f"row scales {r}")
        assert out["g_row"] == d
    cols = np.sort(rng.choice(C, 32, replace=False))
    z = Q.rht16(np.ascontiguousarray(x32[:, cols].T), signs)
    Ac = out["amax_rht"]
    # the rotated amax is global: pin it on a slab bound and recompute codes with the GPU-independent value
    ref_Ac = max(float(Q.amax(Q.rht16(np.ascontiguousarray(x32[:, c:c + 512].T), signs))) for c in range(0, C, 512))
    assert float(Ac) == ref_Ac
    for i, c in enumerate(cols):
        q, s, d = Q.nvfp4_quantize(z[i:i + 1], np.float32(ref_Ac),
                                   sr=dict(seed=seed, copy_id=1, offset=offset, row0=int(c), cols=R))
        G.assert_equal_codes(out["q_col"][c:c + 1], q, f"col {c}")
        G.assert_equal_codes(out["s_col"][c:c + 1], s, f"col scales {c}")


def test_nvfp4_weight_2d_codonfm():
    w = gaussian((4096, 4096), 0.02, 81).to(G.DEV)
    out = G.nvfp4(w, te.NVFP4_2D)
    G.assert_equal_codes(out["q_col"], out["q_row"].T, "2D transpose consistency")
    x32 = G.f32_np(w)
    q, s, d = Q.nvfp4_quantize(x32[:256], Q.amax(x32), block2d=True)
    G.assert_equal_codes(out["q_row"][:256], q, "rows 0..255")
    G.assert_equal_codes(out["s_row"][:256], s, "scales 0..255")
