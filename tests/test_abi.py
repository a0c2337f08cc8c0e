"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function that include/nvfp4.h declares, and rejects bad arguments before it
touches a device."""
import ctypes
import os
import re

import pytest

import nvfp4_block_scaled_27_b300 as nv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_27_b300 import _build
    _build.build()
    return nv.load_library()


def test_header_declares_the_three_hot_path_calls():
    decl = _declared_functions()
    for name in ("nvfp4_quantize", "nvfp4_quantize_rht_sr", "nvfp4_gemm"):
        assert name in decl


def test_library_exports_every_declared_symbol(lib):
    decl = _declared_functions()
    assert decl, "no declarations parsed"
    for name in decl:
        assert hasattr(lib, name), f"missing export {name}"
    assert set(decl) == set(nv.EXPORTED)


def test_scales_bytes(lib):
    assert nv.scales_bytes(256, 256, nv.SCALES_CANONICAL) == 256 * 16
    assert nv.scales_bytes(256, 256, nv.SCALES_MMA) == 256 * 16
    assert nv.scales_bytes(130, 64, nv.SCALES_MMA) == 256 * 4      # rows padded to 128
    assert nv.scales_bytes(130, 64, nv.SCALES_CANONICAL) == 130 * 4
    assert nv.scales_bytes(16, 48, nv.SCALES_MMA) == 0             # cols % 64 != 0
    assert nv.scales_bytes(16, 40, nv.SCALES_CANONICAL) == 0       # cols % 16 != 0
    assert nv.scales_bytes(16, 64, 7) == 0


def test_status_strings_and_version(lib):
    for code in (nv.OK, nv.ERR_INVALID_ARG, nv.ERR_UNSUPPORTED, nv.ERR_CUDA, nv.ERR_TIMEOUT, nv.ERR_NONFINITE):
        s = lib.nvfp4_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.nvfp4_status_string(12345).decode() == "unknown status"
    assert lib.nvfp4_version() >= 100


def test_invalid_arguments_rejected_on_host(lib):
    # null output descriptor, unknown flags, bad shapes: refused before any
    # device work
    assert lib.nvfp4_quantize(None, 16, 16, 16, 0, 0, None, None, None) == nv.ERR_INVALID_ARG
    t = nv.CTensor(1, 1, 1, 1, 16, 16, nv.SCALES_CANONICAL, 0)
    assert lib.nvfp4_quantize(16, 16, 16, 16, 0x80, 0, None, ctypes.byref(t), None) == nv.ERR_INVALID_ARG
    t_bad = nv.CTensor(1, 1, 1, 1, 16, 24, nv.SCALES_CANONICAL, 0)  # cols % 16 != 0
    assert lib.nvfp4_quantize(16, 16, 24, 24, 0, 0, None, ctypes.byref(t_bad), None) == nv.ERR_INVALID_ARG
    t_shape = nv.CTensor(1, 1, 1, 1, 32, 16, nv.SCALES_CANONICAL, 0)  # wrong output shape
    assert lib.nvfp4_quantize(16, 16, 16, 16, 0, 0, None, ctypes.byref(t_shape), None) == nv.ERR_INVALID_ARG
    # RHT with 2D blocks is not a mode
    assert lib.nvfp4_quantize_rht_sr(16, 16, 16, 16, nv.BLOCK_2D, 0, 0, None, ctypes.byref(t), None) \
        == nv.ERR_INVALID_ARG
    # GEMM: canonical scales, K mismatch, K % 256
    a = nv.CTensor(16, 16, 16, 16, 128, 256, nv.SCALES_CANONICAL, 0)
    b = nv.CTensor(16, 16, 16, 16, 128, 256, nv.SCALES_MMA, 0)
    assert lib.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 16, 128, None) == nv.ERR_INVALID_ARG
    a2 = nv.CTensor(16, 16, 16, 16, 128, 512, nv.SCALES_MMA, 0)
    assert lib.nvfp4_gemm(ctypes.byref(a2), ctypes.byref(b), 16, 128, None) == nv.ERR_INVALID_ARG
    a3 = nv.CTensor(16, 16, 16, 16, 128, 192, nv.SCALES_MMA, 0)
    b3 = nv.CTensor(16, 16, 16, 16, 128, 192, nv.SCALES_MMA, 0)
    assert lib.nvfp4_gemm(ctypes.byref(a3), ctypes.byref(b3), 16, 128, None) == nv.ERR_INVALID_ARG
    # ldc below N
    assert lib.nvfp4_gemm(ctypes.byref(b), ctypes.byref(b), 16, 64, None) == nv.ERR_INVALID_ARG


def test_gemm_group_arguments_rejected_on_host(lib):
    """Count out of range, null arrays, and one bad problem among good ones:
    nothing is launched (no device is needed to reach these rejections)."""
    good = nv.CTensor(16, 16, 16, 16, 128, 256, nv.SCALES_MMA, 0)
    bad = nv.CTensor(16, 16, 16, 16, 128, 256, nv.SCALES_CANONICAL, 0)
    P = ctypes.c_void_p
    a = (P * 2)(ctypes.addressof(good), ctypes.addressof(good))
    b = (P * 2)(ctypes.addressof(good), ctypes.addressof(bad))
    c = (P * 2)(16, 16)
    ld = (ctypes.c_int64 * 2)(128, 128)
    cast = lambda arr: ctypes.cast(arr, P)  # noqa: E731
    assert lib.nvfp4_gemm_group(0, cast(a), cast(a), cast(c), cast(ld), None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm_group(3, cast(a), cast(a), cast(c), cast(ld), None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm_group(2, None, cast(a), cast(c), cast(ld), None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm_group(2, cast(a), cast(a), cast(c), None, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_gemm_group(2, cast(a), cast(b), cast(c), cast(ld), None) == nv.ERR_INVALID_ARG  # 2nd bad
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_gemm_group([])


def test_dual_and_mxfp4_arguments_rejected_on_host(lib):
    row = nv.CTensor(1, 1, 1, 1, 64, 256, nv.SCALES_MMA, 0)
    col = nv.CTensor(1, 1, 1, 1, 256, 64, nv.SCALES_MMA, 0)
    ok_args = (16, 64, 256, 256)
    # 2D blocks / transposition are not row modes of the dual call
    assert lib.nvfp4_quantize_dual(*ok_args, nv.BLOCK_2D, 0, 0, 0, None, None, ctypes.byref(row), ctypes.byref(col),
                                   None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_dual(*ok_args, nv.TRANSPOSE_OUT, 0, 0, 0, None, None, ctypes.byref(row),
                                   ctypes.byref(col), None) == nv.ERR_INVALID_ARG
    # output shapes swapped, mixed scale layouts, rows % 64 for the MMA layout
    assert lib.nvfp4_quantize_dual(*ok_args, 0, 0, 0, 0, None, None, ctypes.byref(col), ctypes.byref(row), None) \
        == nv.ERR_INVALID_ARG
    col_c = nv.CTensor(1, 1, 1, 1, 256, 64, nv.SCALES_CANONICAL, 0)
    assert lib.nvfp4_quantize_dual(*ok_args, 0, 0, 0, 0, None, None, ctypes.byref(row), ctypes.byref(col_c), None) \
        == nv.ERR_INVALID_ARG
    row48 = nv.CTensor(1, 1, 1, 1, 48, 256, nv.SCALES_MMA, 0)
    col48 = nv.CTensor(1, 1, 1, 1, 256, 48, nv.SCALES_MMA, 0)
    assert lib.nvfp4_quantize_dual(16, 48, 256, 256, 0, 0, 0, 0, None, None, ctypes.byref(row48), ctypes.byref(col48),
                                   None) == nv.ERR_INVALID_ARG
    # MXFP4: cols % 32, ld < cols, ld % 8
    assert lib.nvfp4_quantize_mxfp4(16, 4, 48, 48, 16, 16, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_mxfp4(16, 4, 64, 32, 16, 16, None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_mxfp4(16, 4, 64, 68, 16, 16, None) == nv.ERR_INVALID_ARG


def test_mma_rate_probe_arguments_rejected_on_host(lib):
    pairs = ctypes.c_int32(0)
    assert lib.nvfp4_mma_rate_probe(0, 256, 16, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_mma_rate_probe((1 << 20) + 1, 256, 16, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_mma_rate_probe(64, 192, 16, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_mma_rate_probe(64, 256, None, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG
    assert lib.nvfp4_mma_rate_probe(64, 256, 12, ctypes.byref(pairs), None) == nv.ERR_INVALID_ARG  # misaligned
    assert lib.nvfp4_mma_rate_probe(64, 256, 16, None, None) == nv.ERR_INVALID_ARG
    assert pairs.value == 0


def test_copy_rate_probe_arguments_rejected_on_host(lib):
    ok = (256, 1 << 20, 0, 4, 16, 16, None)
    bad = [
        (None, 1 << 20, 0, 4, 16, 16, None),
        (256, 16383, 0, 4, 16, 16, None),          # under one chunk
        (256, 262143, 1, 4, 16, 16, None),         # under one 128-row band of boxes
        (256, 1 << 20, 2, 4, 16, 16, None),        # unknown mode
        (256, 1 << 20, 0, 0, 16, 16, None),
        (256, 1 << 20, 0, 4, 0, 16, None),
        (256, 1 << 20, 0, 4, (1 << 20) + 1, 16, None),
        (264, 1 << 20, 0, 4, 16, 16, None),        # src misaligned
        (256, 1 << 20, 0, 4, 16, 12, None),        # out misaligned
        (256, 1 << 20, 0, 4, 16, None, None),
    ]
    assert len(ok) == len(bad[0])
    for args in bad:
        assert lib.nvfp4_copy_rate_probe(*args) == nv.ERR_INVALID_ARG, args


def test_compute_calls_refuse_cpu_tensors():
    import torch
    x = torch.zeros(16, 16, dtype=torch.bfloat16)
    with pytest.raises(nv.Nvfp4Error):
        nv.quantize(x, layout=nv.SCALES_CANONICAL)
