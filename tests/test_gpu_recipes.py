"""DelayedScaling end to end on the GPU against the oracle.

1. The 768 -> 768 linear of the FP8 tutorial (X [1024, 768] fp32 ~ U[0,1),
   re-drawn every step), HYBRID recipe, history 16, algo max, margin 0: twenty
   steps of Fprop / Dgrad / Wgrad with the scales the history dictates.  Codes,
   amaxes, histories, scales and scale_invs bit-exact; GEMM outputs within 1e-3.
2. A multi-layer schedule (4 layers x 4 linears x 3 passes, reduced sizes) with
   Student-t(3) activations carrying 0.1 % outliers x100 and a per-step power of
   two on every tensor, so that amaxes move, histories wrap (L = 16) or keep
   growing (L = 1024), and delayed scales saturate the outliers.  Histories and
   scales bit-exact after every step.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from oracle import formats as F
from oracle import quantize as Q
from oracle import recipes as Rc
from synthetic import gaussian, linear768, student_t_outliers
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().numpy().view(np.uint32)


def test_linear768_delayed_scaling_20_steps():
    L = 16
    recipe = te.te_recipe(te.E4M3, te.E5M2, L, te.ALGO_MAX, 0, 1)
    dev = G.DEV
    # device recipe state: forward tensors (X, W), backward (dY)
    fwd = dict(hist=torch.zeros(2 * L, device=dev), scale=torch.ones(2, device=dev),
               sinv=torch.ones(2, device=dev), amax=torch.zeros(2, device=dev))
    bwd = dict(hist=torch.zeros(L, device=dev), scale=torch.ones(1, device=dev),
               sinv=torch.ones(1, device=dev), amax=torch.zeros(1, device=dev))
    ox = Rc.DelayedScalingState("e4m3", L)
    ow = Rc.DelayedScalingState("e4m3", L)
    od = Rc.DelayedScalingState("e5m2", L)
    saturated_steps = 0
    for t in range(20):
        x, w, b, dy = linear768(t)
        x32, w32, dy32 = x.numpy(), w.numpy(), dy.numpy()
        X, W, B, DY = x.to(dev), w.to(dev), b.to(dev), dy.to(dev)
        M, K = X.shape
        N = W.shape[0]
        xr, xc = G.u8(M, K), G.u8(K, M)
        wr, wc = G.u8(N, K), G.u8(K, N)
        dr, dc = G.u8(M, N), G.u8(N, M)
        te.te_quantize_fp8(X, te.E4M3, fwd["scale"][0:1], 0, xr, xc, fwd["amax"][0:1])
        te.te_quantize_fp8(W, te.E4M3, fwd["scale"][1:2], 0, wr, wc, fwd["amax"][1:2])
        te.te_quantize_fp8(DY, te.E5M2, bwd["scale"][0:1], 0, dr, dc, bwd["amax"][0:1])
        Y = torch.empty(M, N, dtype=torch.float32, device=dev)
        DX = torch.empty(M, K, dtype=torch.float32, device=dev)
        DW = torch.empty(N, K, dtype=torch.float32, device=dev)
        te.te_gemm_fp8(xr, te.E4M3, wr, te.E4M3, fwd["sinv"][0:1], fwd["sinv"][1:2], Y, B)
        te.te_gemm_fp8(dr, te.E5M2, wc, te.E4M3, bwd["sinv"][0:1], fwd["sinv"][1:2], DX)
        te.te_gemm_fp8(dc, te.E5M2, xc, te.E4M3, bwd["sinv"][0:1], fwd["sinv"][0:1], DW)
        torch.cuda.synchronize()
        # oracle: quantize with the scales in use at this step
        eq = {}
        for name, arr, st, fmt in (("x", x32, ox, "e4m3"), ("w", w32, ow, "e4m3"), ("dy", dy32, od, "e5m2")):
            eq[name] = Q.fp8_quantize(arr, st.scale, fmt) + (st.scale_inv,)
        G.assert_equal_codes(xr.cpu().numpy(), eq["x"][0], f"X row step {t}")
        G.assert_equal_codes(xc.cpu().numpy(), eq["x"][1], f"X col step {t}")
        G.assert_equal_codes(wr.cpu().numpy(), eq["w"][0], f"W row step {t}")
        G.assert_equal_codes(dc.cpu().numpy(), eq["dy"][1], f"dY col step {t}")
        assert fwd["amax"][0].item() == Q.amax(x32) and bwd["amax"][0].item() == Q.amax(dy32)
        saturated_steps += int(np.any(np.abs(F.decode(eq["x"][0], "e4m3")) == 448.0))

        def deq(q, si, fmt):
            return Q.fp8_dequant(q, si, fmt)
        ops = ((Y, deq(eq["x"][0], ox.scale_inv, "e4m3"), deq(eq["w"][0], ow.scale_inv, "e4m3"), b.numpy(), "Y"),
               (DX, deq(eq["dy"][0], od.scale_inv, "e5m2"), deq(eq["w"][1], ow.scale_inv, "e4m3"), None, "dX"),
               (DW, deq(eq["dy"][1], od.scale_inv, "e5m2"), deq(eq["x"][1], ox.scale_inv, "e4m3"), None, "dW"))
        for got, a64, b64, bias, nm in ops:
            G.check_gemm(got.cpu().numpy(), a64, b64, bias=bias, what=f"{nm} step {t}")
        # end of step: record amaxes, refresh scales
        te.te_scale_update(recipe, 0, fwd["hist"], fwd["amax"], fwd["scale"], fwd["sinv"], t)
        te.te_scale_update(recipe, 1, bwd["hist"], bwd["amax"], bwd["scale"], bwd["sinv"], t)
        ox.update(Q.amax(x32), t)
        ow.update(Q.amax(w32), t)
        od.update(Q.amax(dy32), t)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(fwd["scale"]), np.array([ox.scale, ow.scale], np.float32).view(np.uint32))
        np.testing.assert_array_equal(_bits(fwd["sinv"]), np.array([ox.scale_inv, ow.scale_inv], np.float32).view(np.uint32))
        np.testing.assert_array_equal(_bits(bwd["scale"]), np.array([od.scale], np.float32).view(np.uint32))
        np.testing.assert_array_equal(_bits(fwd["hist"]).reshape(2, L), np.stack([ox.hist, ow.hist]).view(np.uint32))
        np.testing.assert_array_equal(_bits(bwd["hist"]), od.hist.view(np.uint32))
    assert ox.scale != 1.0 and od.scale != 1.0
    G.check_no_device_error()


@pytest.mark.parametrize("L", [16, 1024])
def test_multilayer_schedule_student_t(L):
    layers, M, h, f = 4, 512, 256, 1024
    steps = 24 if L == 16 else 20
    dev = G.DEV
    shapes = [(h, 3 * h), (h, h), (h, f), (f, h)]          # (in, out) of the four linears
    n_lin = layers * len(shapes)
    recipe = te.te_recipe(te.E4M3, te.E5M2, L, te.ALGO_MAX, 0, 1)
    fwd = dict(hist=torch.zeros(2 * n_lin * L, device=dev), scale=torch.ones(2 * n_lin, device=dev),
               sinv=torch.ones(2 * n_lin, device=dev), amax=torch.zeros(2 * n_lin, device=dev))
    bwd = dict(hist=torch.zeros(n_lin * L, device=dev), scale=torch.ones(n_lin, device=dev),
               sinv=torch.ones(n_lin, device=dev), amax=torch.zeros(n_lin, device=dev))
    o_fwd = [Rc.DelayedScalingState("e4m3", L) for _ in range(2 * n_lin)]
    o_bwd = [Rc.DelayedScalingState("e5m2", L) for _ in range(n_lin)]
    base = []
    for i in range(n_lin):
        k_in, n_out = shapes[i % len(shapes)]
        base.append((student_t_outliers((M, k_in), 7000 + i, dtype=torch.float32),
                     gaussian((n_out, k_in), 0.02, 8000 + i, dtype=torch.float32),
                     gaussian((M, n_out), 1e-3, 9000 + i, dtype=torch.float32)))
    rng = np.random.default_rng(L)
    saw_saturation = False
    for t in range(steps):
        k = rng.integers(-3, 4, size=(n_lin, 3))          # per-step power of two per tensor (exact)
        amx = np.zeros((n_lin, 3), np.float32)
        for i, (x0, w0, d0) in enumerate(base):
            tensors = [x0 * 2.0 ** int(k[i, 0]), w0 * 2.0 ** int(k[i, 1]), d0 * 2.0 ** int(k[i, 2])]
            for j, (tt, fmt, slot) in enumerate(((tensors[0], te.E4M3, ("f", 2 * i)), (tensors[1], te.E4M3, ("f", 2 * i + 1)),
                                                  (tensors[2], te.E5M2, ("b", i)))):
                st = fwd if slot[0] == "f" else bwd
                idx = slot[1]
                T = tt.to(dev)
                R, C = T.shape
                qr = G.u8(R, C)
                te.te_quantize_fp8(T, fmt, st["scale"][idx:idx + 1], 0, qr, None, st["amax"][idx:idx + 1])
                a = Q.amax(tt.numpy())
                amx[i, j] = a
                if i == 0 and j == 0:
                    torch.cuda.synchronize()
                    osc = o_fwd[0].scale
                    G.assert_equal_codes(qr.cpu().numpy(), Q.fp8_cast(tt.numpy(), osc, "e4m3"), f"layer0 X step {t}")
                    saw_saturation |= bool(np.any(qr.cpu().numpy() & 0x7F == 0x7E))
        te.te_scale_update(recipe, 0, fwd["hist"], fwd["amax"], fwd["scale"], fwd["sinv"], t)
        te.te_scale_update(recipe, 1, bwd["hist"], bwd["amax"], bwd["scale"], bwd["sinv"], t)
        for i in range(n_lin):
            o_fwd[2 * i].update(amx[i, 0], t)
            o_fwd[2 * i + 1].update(amx[i, 1], t)
            o_bwd[i].update(amx[i, 2], t)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(fwd["amax"]), amx[:, :2].reshape(-1).view(np.uint32))
        np.testing.assert_array_equal(_bits(fwd["scale"]), np.array([s.scale for s in o_fwd], np.float32).view(np.uint32))
        np.testing.assert_array_equal(_bits(bwd["scale"]), np.array([s.scale for s in o_bwd], np.float32).view(np.uint32))
        np.testing.assert_array_equal(_bits(fwd["sinv"]), np.array([s.scale_inv for s in o_fwd], np.float32).view(np.uint32))
    np.testing.assert_array_equal(_bits(fwd["hist"]).reshape(2 * n_lin, L), np.stack([s.hist for s in o_fwd]).view(np.uint32))
    np.testing.assert_array_equal(_bits(bwd["hist"]).reshape(n_lin, L), np.stack([s.hist for s in o_bwd]).view(np.uint32))
    assert saw_saturation
    G.check_no_device_error()
