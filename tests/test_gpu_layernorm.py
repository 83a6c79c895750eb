"""LayerNorm fused with the FP8 cast of its output, against the oracle.

mu and rsigma against the fp64 definition (fp32 sums of up to 8192 terms: relative
error well under 1e-5); the bf16 LN output within one bf16 rounding of the fp64
value (plus the fp32 arithmetic's few ulps); the FP8 codes bit-exact against the
oracle's cast of the kernel's own bf16 outputs (both decide in fp32) and the amax
exact over them.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from oracle import formats as F
from oracle import quantize as Q
from oracle.layernorm import layernorm
from synthetic import gaussian, student_t_outliers
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,fmt", [(64, 256, "e4m3"), (200 - 8, 768, "e4m3"), (16, 4096, "e5m2"),
                                           (1024, 4096, "e4m3"), (32, 8192, "e4m3"), (48, 48, "e5m2")])
def test_layernorm_fp8(rows, cols, fmt):
    x = student_t_outliers((rows, cols), 900 + cols, dtype=torch.bfloat16).to(G.DEV)
    gamma = (1.0 + gaussian((cols,), 0.1, 901, dtype=torch.float32)).to(G.DEV)
    beta = gaussian((cols,), 0.1, 902, dtype=torch.float32).to(G.DEV)
    eps = 1e-5
    scale_v = 2.0 ** 5 if fmt == "e4m3" else 2.0 ** 12
    code = te.E4M3 if fmt == "e4m3" else te.E5M2
    q = G.u8(rows, cols)
    ln = torch.empty(rows, cols, dtype=torch.bfloat16, device=G.DEV)
    mu, rs = torch.empty(rows, device=G.DEV), torch.empty(rows, device=G.DEV)
    amax, sinv = G.scalar(-1.0), G.scalar(-1.0)
    te.te_layernorm_fp8(x, gamma, beta, eps, code, G.scalar(scale_v), q, ln, mu, rs, amax, sinv)
    torch.cuda.synchronize()
    y64, mu64, rs64 = layernorm(G.f32_np(x), gamma.cpu().numpy(), beta.cpu().numpy(), eps)
    np.testing.assert_allclose(mu.cpu().numpy(), mu64, rtol=1e-5, atol=1e-6 * np.abs(G.f32_np(x)).max())
    np.testing.assert_allclose(rs.cpu().numpy(), rs64, rtol=1e-5)
    ln32 = G.f32_np(ln).astype(np.float64)
    ulp = np.maximum(np.abs(y64), 2.0 ** -126) * 2.0 ** -8          # one bf16 ulp (relative)
    assert np.all(np.abs(ln32 - y64) <= ulp + 1e-5 * np.abs(y64) + 1e-6), float(np.max(np.abs(ln32 - y64) / ulp))
    G.assert_equal_codes(q.cpu().numpy(), Q.fp8_cast(G.f32_np(ln), scale_v, fmt), "LN FP8 codes")
    assert np.float32(amax.item()) == Q.amax(G.f32_np(ln))
    assert np.float32(sinv.item()) == np.float32(1.0) / np.float32(scale_v)
    G.check_no_device_error()


def test_layernorm_rejects_and_optional_outputs():
    x = gaussian((32, 256), 1.0, 5, dtype=torch.bfloat16).to(G.DEV)
    g, b = torch.ones(256, device=G.DEV), torch.zeros(256, device=G.DEV)
    q = G.u8(32, 256)
    te.te_layernorm_fp8(x, g, b, 1e-5, te.E4M3, G.scalar(1.0), q)   # only the FP8 copy
    torch.cuda.synchronize()
    y64, _, _ = layernorm(G.f32_np(x), np.ones(256), np.zeros(256), 1e-5)
    assert np.mean(F.decode(q.cpu().numpy(), "e4m3") == 0) < 0.2
    with pytest.raises(te.TEError):
        te.te_layernorm_fp8(x.float(), g, b, 1e-5, te.E4M3, G.scalar(1.0), q)     # bf16 input only
    with pytest.raises(te.TEError):
        te.te_layernorm_fp8(x, g, b, -1.0, te.E4M3, G.scalar(1.0), q)             # eps must be >= 0
    G.check_no_device_error()


@pytest.mark.parametrize("rows,cols", [(15872, 4096), (15872, 2048), (2048, 8192)])
def test_layernorm_fp8_many_rows_per_group(rows, cols):
    """Enough rows that every row group (register kernel) or warp (shared-memory kernel, 8192
    columns) walks several rows, so the row loop's reuse of its buffers and barriers is exercised:
    sampled rows against the oracle, every FP8 code against the oracle's cast of the kernel's own
    bf16 output, the amax over all of it."""
    x = student_t_outliers((rows, cols), 77 + cols, dtype=torch.bfloat16).to(G.DEV)
    gamma = (1.0 + gaussian((cols,), 0.1, 78, dtype=torch.float32)).to(G.DEV)
    beta = gaussian((cols,), 0.1, 79, dtype=torch.float32).to(G.DEV)
    eps, scale_v = 1e-5, 2.0 ** 5
    q = G.u8(rows, cols)
    ln = torch.empty(rows, cols, dtype=torch.bfloat16, device=G.DEV)
    mu, rs = torch.empty(rows, device=G.DEV), torch.empty(rows, device=G.DEV)
    amax = G.scalar(-1.0)
    te.te_layernorm_fp8(x, gamma, beta, eps, te.E4M3, G.scalar(scale_v), q, ln, mu, rs, amax)
    torch.cuda.synchronize()
    G.check_no_device_error()
    rng = np.random.default_rng(rows + cols)
    idx = np.unique(np.concatenate([rng.choice(rows, 256, replace=False), [0, 1, rows - 2, rows - 1]]))
    x32 = G.f32_np(x[torch.from_numpy(idx).to(G.DEV)])
    y64, mu64, rs64 = layernorm(x32, gamma.cpu().numpy(), beta.cpu().numpy(), eps)
    np.testing.assert_allclose(mu.cpu().numpy()[idx], mu64, rtol=1e-5, atol=1e-6 * np.abs(x32).max())
    np.testing.assert_allclose(rs.cpu().numpy()[idx], rs64, rtol=1e-5)
    ln_s = G.f32_np(ln[torch.from_numpy(idx).to(G.DEV)]).astype(np.float64)
    ulp = np.maximum(np.abs(y64), 2.0 ** -126) * 2.0 ** -8
    assert np.all(np.abs(ln_s - y64) <= ulp + 1e-5 * np.abs(y64) + 1e-6)
    ln32 = G.f32_np(ln)
    G.assert_equal_codes(q.cpu().numpy(), Q.fp8_cast(ln32, scale_v, "e4m3"), "LN FP8 codes, all rows")
    assert np.float32(amax.item()) == Q.amax(ln32)
