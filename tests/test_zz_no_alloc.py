"""The allocation-free bias-gradient quantization (for callers that cannot allocate
device memory at that point) gives exactly what the workspace entry point gives.

Collected last on purpose.  Two calls in a row with different inputs: the second
must not be affected by what the first left in the library's shared scratch array.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from synthetic import gaussian
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _run(fn_noalloc, dy, current):
    rows, cols = dy.shape
    q_row, q_col = G.u8(rows, cols), G.u8(cols, rows)
    amax, sinv = G.scalar(-1.0), G.scalar(-1.0)
    dbias = torch.full((cols,), float("nan"), device=G.DEV)
    scale = None if current else G.scalar(2.0 ** 13)
    if fn_noalloc:
        te.te_quantize_fp8_dbias_noalloc(dy, te.E5M2, dbias, scale=scale, compute_scale=current, q_row=q_row,
                                         q_col=q_col, amax_out=amax, scale_inv_out=sinv)
    else:
        ws = torch.empty(te.te_dbias_workspace_bytes(rows, cols) // 4, device=G.DEV)
        te.te_quantize_fp8_dbias(dy, te.E5M2, dbias, ws, scale=scale, compute_scale=current, q_row=q_row,
                                 q_col=q_col, amax_out=amax, scale_inv_out=sinv)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (q_row, q_col, amax, sinv, dbias)]


@pytest.mark.parametrize("current", [0, 1])
def test_noalloc_matches_workspace_entry_point_on_two_calls(current):
    shapes = [(15872, 4096), (512, 1008)]          # the largest allowed CodonFM dY, then a small one
    for i, (rows, cols) in enumerate(shapes):
        dy = gaussian((rows, cols), 1e-3, 31 + i, dtype=torch.bfloat16).to(G.DEV)
        got = _run(True, dy, current)
        ref = _run(False, dy, current)
        for g, r, name in zip(got, ref, ("q_row", "q_col", "amax", "scale_inv", "dbias")):
            # same kernels and the same fixed summation order: identical bits
            np.testing.assert_array_equal(g.view(np.uint8), r.view(np.uint8), err_msg=f"call {i}: {name}")
    G.check_no_device_error()


def test_noalloc_allocates_no_device_memory():
    # after a first call (which looks up the array's address), further calls change neither
    # torch's allocator count nor the device's free memory
    rows, cols = 4096, 2048
    dy = gaussian((rows, cols), 1e-3, 77, dtype=torch.bfloat16).to(G.DEV)
    q_col, dbias, sinv = G.u8(cols, rows), torch.zeros(cols, device=G.DEV), G.scalar()
    scale = G.scalar(2.0 ** 13)

    def call():
        te.te_quantize_fp8_dbias_noalloc(dy, te.E5M2, dbias, scale=scale, q_col=q_col, scale_inv_out=sinv)

    call()
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    G.check_no_device_error()


def test_noalloc_rejects_more_partial_sums_than_the_scratch_holds():
    dy = torch.zeros(15872, 16384, dtype=torch.bfloat16, device=G.DEV)   # 248 x 16384 partial sums > 2^20
    dbias = torch.zeros(16384, device=G.DEV)
    with pytest.raises(te.TEError) as e:
        te.te_quantize_fp8_dbias_noalloc(dy, te.E5M2, dbias, scale=G.scalar(1.0), q_col=G.u8(16384, 15872))
    assert e.value.status == 2   # TE_ERR_SHAPE, before anything is enqueued
    G.check_no_device_error()
