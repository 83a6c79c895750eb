"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point declared in include/te_gb300.h, validates arguments before
touching the device, and its block-scale layout helpers match an independent
restatement of the tensor-core scale layout."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "te_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_precision_transformer_gb300 import build, _lib
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:te_status|size_t|const char\*|uint64_t)\s+(te_\w+)\s*\(", txt, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 14
    from nvfp4_precision_transformer_gb300 import _lib
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, n


def test_status_strings(lib):
    for s in range(9):
        assert lib.te_status_str(s).startswith(b"TE_")


def test_validation_before_any_device_work(lib):
    from nvfp4_precision_transformer_gb300 import _lib as L
    fake = ctypes.c_void_p(0x1000)       # never dereferenced: validation fails first
    # rows not a multiple of 16
    assert lib.te_quantize_fp8(fake, L.BF16, 24, 32, L.E4M3, fake, 0, None, None, None, None, None) == 2
    # bad dtype
    assert lib.te_quantize_fp8(fake, L.E2M1, 32, 32, L.E4M3, fake, 0, None, None, None, None, None) == 4
    assert lib.te_quantize_fp8(fake, L.BF16, 32, 32, L.E2M1, fake, 0, None, None, None, None, None) == 4
    # current scaling without amax_out
    assert lib.te_quantize_fp8(fake, L.BF16, 32, 32, L.E4M3, None, 1, None, None, None, None, None) == 1
    # misaligned input
    assert lib.te_amax_reduce(ctypes.c_void_p(0x1004), L.BF16, 32, 32, fake, None, 0, None) == 3
    # mxfp8 col copy needs rows % 32
    assert lib.te_quantize_mxfp8(fake, L.BF16, 48, 64, None, None, fake, fake, None) == 2
    # nvfp4: 2D with RHT is rejected; unknown flag
    assert lib.te_quantize_nvfp4(fake, L.BF16, 32, 32, 3, 0, 0, 0, fake, fake, fake, fake, fake,
                                 None, None, None, None) == 8
    assert lib.te_quantize_nvfp4(fake, L.BF16, 32, 32, 8, 0, 0, 0, fake, fake, fake, fake, fake,
                                 None, None, None, None) == 8
    # GEMMs: shapes, K == 0, dtype
    assert lib.te_gemm_bf16(fake, 0, fake, 0, None, fake, L.BF16, 0, 32, 40, 32, None) == 2
    assert lib.te_gemm_bf16(fake, 0, fake, 0, None, fake, L.BF16, 0, 32, 32, 0, None) == 2
    assert lib.te_gemm_bf16(fake, 2, fake, 0, None, fake, L.BF16, 0, 32, 32, 32, None) == 8
    assert lib.te_gemm_fp8(fake, L.E2M1, fake, L.E4M3, fake, fake, None, fake, L.BF16, 0, 32, 32, 32, None) == 4
    assert lib.te_gemm_nvfp4(fake, fake, fake, fake, fake, fake, None, fake, L.BF16, 0, 32, 32, 48, None) == 2
    assert lib.te_gemm_mxfp8(fake, L.E4M3, fake, fake, L.E4M3, fake, None, fake, L.E8M0, 0, 32, 32, 32, None) == 4
    # accumulate adds into an fp32 D only; any flag other than 0 / 1 is rejected
    assert lib.te_gemm_fp8(fake, L.E4M3, fake, L.E4M3, fake, fake, None, fake, L.BF16, 1, 32, 32, 32, None) == 4
    assert lib.te_gemm_bf16(fake, 0, fake, 0, None, fake, L.F32, 2, 32, 32, 32, None) == 8
    # empty GEMM is a no-op success
    assert lib.te_gemm_bf16(None, 0, None, 0, None, None, L.BF16, 0, 0, 32, 32, None) == 0
    # the allocation-free dbias quantization validates before it looks anything up on a device
    assert lib.te_quantize_fp8_dbias_noalloc(fake, L.BF16, 24, 32, L.E5M2, fake, 0, None, fake, None, None,
                                             fake, None) == 2
    assert lib.te_quantize_fp8_dbias_noalloc(fake, L.BF16, 32, 32, L.E2M1, fake, 0, None, fake, None, None,
                                             fake, None) == 4
    assert lib.te_quantize_fp8_dbias_noalloc(fake, L.BF16, 32, 32, L.E5M2, None, 0, None, fake, None, None,
                                             fake, None) == 1
    assert lib.te_quantize_fp8_dbias_noalloc(fake, L.BF16, 32, 32, L.E5M2, fake, 0, None, fake, None, None,
                                             ctypes.c_void_p(0x1002), None) == 3
    assert lib.te_quantize_fp8_dbias_noalloc(fake, L.BF16, 15872, 16384, L.E5M2, fake, 0, None, fake, None, None,
                                             fake, None) == 2     # more partial sums than the fixed array holds
    # recipe validation
    r = L.te_recipe(L.E4M3, L.E5M2, 0, 0, 0, 1)
    assert lib.te_scale_update(ctypes.byref(r), 0, 4, fake, fake, fake, fake, 0, None) == 8
    r = L.te_recipe(L.E4M3, L.E2M1, 16, 0, 0, 1)
    assert lib.te_scale_update(ctypes.byref(r), 1, 4, fake, fake, fake, fake, 0, None) == 4


def _offset(r, j, kpad):
    # tensor-core block-scale layout: 128 x 4 tiles of 512 bytes, tile-major
    tile = (r // 128) * (kpad // 4) + j // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (j % 4)


@pytest.mark.parametrize("fmt,blk,padk", [(5, 32, 4), (6, 16, 16)])
@pytest.mark.parametrize("rows,cols", [(128, 128), (48, 96), (256, 512), (16, 32)])
def test_scale_layout_helpers(lib, fmt, blk, padk, rows, cols):
    from nvfp4_precision_transformer_gb300 import _lib as L
    nb = cols // blk
    kpad = -(-nb // padk) * padk
    rpad = -(-rows // 128) * 128
    assert L.te_scale_bytes(fmt, rows, cols) == rpad * kpad
    logical = np.random.default_rng(rows + cols).integers(0, 255, size=(rows, nb)).astype(np.uint8)
    sw = np.zeros(rpad * kpad, np.uint8)
    for r in range(rows):
        for j in range(nb):
            sw[_offset(r, j, kpad)] = logical[r, j]
    np.testing.assert_array_equal(L.te_scale_unswizzle(fmt, rows, cols, sw), logical)


def test_scale_bytes_invalid(lib):
    from nvfp4_precision_transformer_gb300 import _lib as L
    assert L.te_scale_bytes(L.E8M0, 32, 48) == 0
    assert L.te_scale_bytes(L.E4M3, 32, 64) == 0
