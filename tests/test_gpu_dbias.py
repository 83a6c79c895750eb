"""Bias gradient fused with the FP8 quantization of dY, against the oracle.

The quantized copies must be bit-identical to te_quantize_fp8's; dbias is the
column sum of dY, computed in fp32 in fixed-order levels (64 rows per tile, the
tiles in 8 strided groups, the 8 group sums), so it is compared with the fp64 sum
within the fp32 summation bound (64 + tiles + 8) * 2^-24 * sum |dY[:, n]|.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from oracle import quantize as Q
from synthetic import gaussian
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols,dtype", [(15872, 4096, torch.bfloat16), (15872 // 8, 4096, torch.bfloat16),
                                             (208, 336, torch.bfloat16),
                                             (64, 64, torch.float32), (96, 48, torch.float32), (16, 16, torch.bfloat16)])
@pytest.mark.parametrize("current", [0, 1])
def test_fp8_dbias_fused(rows, cols, dtype, current):
    dy = gaussian((rows, cols), 1e-3, 4242 + rows, dtype=dtype).to(G.DEV)
    q_row, q_col = G.u8(rows, cols), G.u8(cols, rows)
    amax, sinv = G.scalar(-1.0), G.scalar(-1.0)
    scale = None if current else G.scalar(2.0 ** 14)
    dbias = torch.full((cols,), -7.0, dtype=torch.float32, device=G.DEV)
    ws = torch.full((te.te_dbias_workspace_bytes(rows, cols) // 4,), float("nan"), device=G.DEV)
    te.te_quantize_fp8_dbias(dy, te.E5M2, dbias, ws, scale=scale, compute_scale=current, q_row=q_row, q_col=q_col,
                             amax_out=amax, scale_inv_out=sinv)
    ref_row, ref_col, ref_amax, ref_sinv = G.fp8(dy, te.E5M2, scale=None if current else 2.0 ** 14, current=bool(current))
    torch.cuda.synchronize()
    G.assert_equal_codes(q_row.cpu().numpy(), ref_row, "row copy")
    G.assert_equal_codes(q_col.cpu().numpy(), ref_col, "col copy")
    assert np.float32(amax.item()) == ref_amax and np.float32(sinv.item()) == ref_sinv
    x = G.f32_np(dy).astype(np.float64)
    ref = Q.dbias(x)
    tiles = (rows + 63) // 64
    bound = (64 + tiles + 8) * 2.0 ** -24 * np.abs(x).sum(axis=0) + 1e-30
    got = dbias.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    G.check_no_device_error()


def test_fp8_dbias_row_copy_only_and_empty():
    dy = gaussian((128, 96), 1.0, 9, dtype=torch.bfloat16).to(G.DEV)
    q_row = G.u8(128, 96)
    dbias = torch.zeros(96, device=G.DEV)
    ws = torch.empty(te.te_dbias_workspace_bytes(128, 96) // 4, device=G.DEV)
    te.te_quantize_fp8_dbias(dy, te.E4M3, dbias, ws, scale=G.scalar(1.0), q_row=q_row)
    torch.cuda.synchronize()
    x = G.f32_np(dy).astype(np.float64)
    np.testing.assert_allclose(dbias.cpu().numpy(), Q.dbias(x), rtol=0, atol=(64 + 2 + 8) * 2.0 ** -24 * np.abs(x).sum(0).max())
    # no rows: dbias is zero; a too-small workspace is refused before anything runs
    empty = torch.empty(0, 96, dtype=torch.bfloat16, device=G.DEV)
    d0 = torch.full((96,), 5.0, device=G.DEV)
    te.te_quantize_fp8_dbias(empty, te.E4M3, d0, None, scale=G.scalar(1.0))
    torch.cuda.synchronize()
    assert torch.count_nonzero(d0).item() == 0
    with pytest.raises(te.TEError):
        te.te_quantize_fp8_dbias(dy, te.E4M3, dbias, ws[:10], scale=G.scalar(1.0), q_row=q_row)
    G.check_no_device_error()
