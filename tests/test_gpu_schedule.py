"""The 24-layer DelayedScaling schedule (here 3 layers at reduced sizes): each tensor
quantized once per step into both copies, batched scale updates; histories and
scales bit-exact against the oracle after every step, the last layer's GEMMs within
1e-3, and CUDA-graph replay bit-identical to eager execution."""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from nvfp4_precision_transformer_gb300.linear import ScheduleGraphs, ScheduleStep
from oracle import quantize as Q
from oracle import recipes as Rc
from synthetic import gaussian, student_t_outliers
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

LAYERS, M, H, F = 3, 256, 128, 256
SHAPES = [(H, 3 * H), (H, H), (H, F), (F, H)]


def _inputs():
    out = []
    for l in range(LAYERS):
        lin = []
        for i, (k_in, n_out) in enumerate(SHAPES):
            s = 5000 + 100 * l + 10 * i
            lin.append((student_t_outliers((M, k_in), s, dtype=torch.bfloat16).to(G.DEV),
                        gaussian((n_out, k_in), 0.02, s + 1).to(G.DEV),
                        gaussian((M, n_out), 1e-3, s + 2).to(G.DEV),
                        gaussian((n_out,), 0.02, s + 3, dtype=torch.float32).to(G.DEV)))
        out.append(lin)
    return out


def _perturb(layers, step):
    # an exact power of two per tensor and step moves the amaxes (bf16 scaling by 2^k is exact)
    rng = np.random.default_rng(step)
    for lin in layers:
        for x, w, dy, _ in lin:
            for t in (x, w, dy):
                t.mul_(2.0 ** int(rng.integers(-2, 3)))


def _bits(t):
    return t.detach().cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("L", [16, 4])
def test_schedule_against_oracle_and_graph_replay(L):
    steps = 2 * L + 3                       # histories wrap
    layers_a, layers_b = _inputs(), _inputs()
    sa = ScheduleStep(layers_a, history_len=L)
    ox = [Rc.DelayedScalingState("e4m3", L) for _ in range(2 * 4 * LAYERS)]
    od = [Rc.DelayedScalingState("e5m2", L) for _ in range(4 * LAYERS)]
    for t in range(steps):
        _perturb(layers_a, t)
        # oracle scales in use this step (before the update)
        scales_x = [s.scale for s in ox]
        scales_d = [s.scale for s in od]
        sa.run(t)
        torch.cuda.synchronize()
        k = 0
        for lin in layers_a:
            for x, w, dy, _ in lin:
                ox[2 * k].update(Q.amax(G.f32_np(x)), t)
                ox[2 * k + 1].update(Q.amax(G.f32_np(w)), t)
                od[k].update(Q.amax(G.f32_np(dy)), t)
                k += 1
        np.testing.assert_array_equal(_bits(sa.fwd.scale), np.array([s.scale for s in ox], np.float32).view(np.uint32))
        np.testing.assert_array_equal(_bits(sa.bwd.scale), np.array([s.scale for s in od], np.float32).view(np.uint32))
        np.testing.assert_array_equal(_bits(sa.fwd.hist).reshape(-1, L), np.stack([s.hist for s in ox]).view(np.uint32))
    # last layer's GEMMs of the last step, with the scales that step used
    x, w, dy, b = layers_a[-1][-1]
    k = 4 * LAYERS - 1
    sx, sw, sd = scales_x[2 * k], scales_x[2 * k + 1], scales_d[k]
    x32, w32, dy32 = G.f32_np(x), G.f32_np(w), G.f32_np(dy)
    xr, xc, _, _ = Q.fp8_quantize(x32, sx, "e4m3")
    wr, wc, _, _ = Q.fp8_quantize(w32, sw, "e4m3")
    dr, dc, _, _ = Q.fp8_quantize(dy32, sd, "e5m2")
    isx, isw, isd = (np.float32(1) / np.float32(v) for v in (sx, sw, sd))
    buf = sa.bufs[(x.shape[0], x.shape[1], w.shape[0])]
    ops = {"y": (Q.fp8_dequant(xr, isx, "e4m3"), Q.fp8_dequant(wr, isw, "e4m3"), b.cpu().numpy()),
           "dx": (Q.fp8_dequant(dr, isd, "e5m2"), Q.fp8_dequant(wc, isw, "e4m3"), None),
           "dw": (Q.fp8_dequant(dc, isd, "e5m2"), Q.fp8_dequant(xc, isx, "e4m3"), None)}
    for name, (a64, b64, bias) in ops.items():
        # bf16 outputs against the bf16-rounded fp64 product (and the element-wise bound)
        G.check_gemm(G.f32_np(buf[name]), a64, b64, bias=bias, bf16_out=True, what=name)

    # the same steps with graph replay (one eager step first, as capture requires)
    sb = ScheduleStep(layers_b, history_len=L)
    _perturb(layers_b, 0)
    sb.run(0)
    graphs = ScheduleGraphs(sb)
    for t in range(1, steps):
        _perturb(layers_b, t)
        graphs.run(t)
    torch.cuda.synchronize()
    for a, b2 in ((sa.fwd, sb.fwd), (sa.bwd, sb.bwd)):
        for f in ("hist", "scale", "scale_inv", "amax"):
            np.testing.assert_array_equal(_bits(getattr(a, f)), _bits(getattr(b2, f)))
    for key in sa.bufs:
        for name in ("xr", "xc", "wr", "wc", "dr", "dc", "y", "dx", "dw"):
            assert torch.equal(sa.bufs[key][name], sb.bufs[key][name]), (key, name)
    G.check_no_device_error()
