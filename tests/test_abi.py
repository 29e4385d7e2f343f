"""The C-ABI library loads and exports every declared symbol; argument
validation paths return their status codes (no GPU needed)."""
import ctypes
import os

import pytest

import fp4_block_scaled_e8m0_gb300 as fp4
from fp4_block_scaled_e8m0_gb300 import build as fbuild


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fbuild.lib_path()):
        fbuild.build()
    return fp4.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = fp4.declared_symbols()
    assert len(names) >= 18
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(fp4._SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for s in range(6):
        assert lib.fp4_status_string(s)
    assert b"unsupported" in lib.fp4_status_string(fp4.FP4_ERR_UNSUPPORTED)


def test_scale_buffer_sizes(lib):
    # canonical: one byte per block; MMA layout: rows padded to 128, k to 256
    assert lib.fp4_scales_bytes(8192, 2048, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR, 0) == 8192 * 128
    assert lib.fp4_scales_bytes(8192, 2048, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 0) == 8192 * 128
    assert lib.fp4_scales_bytes(200, 96, fp4.FP4_FMT_MXFP4, fp4.FP4_SF_MMA, 0) == 256 * 8
    assert lib.fp4_scales_bytes(200, 96, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 0) == 256 * 16
    # other blocks: row-major scales only, one byte per block
    assert lib.fp4_scales_bytes(100, 512, fp4.FP4_FMT_MXFP4, fp4.FP4_SF_ROWMAJOR, 128) == 100 * 4
    assert lib.fp4_scales_bytes(100, 512, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR, 64) == 100 * 8
    assert lib.fp4_scales_bytes(100, 512, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 64) == 0
    assert lib.fp4_scales_bytes(100, 512, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR, 48) == 0
    assert lib.fp4_hcp_workspace_bytes(16384, 4096, 369, 2) == 16384 * 768 * 2 + 4096 * 768 * 2
    assert lib.fp4_hcp_select_workspace_bytes(4096) == 4096 * 8


def _fake_ctx():
    # validation runs before the context is touched; a non-null dummy suffices
    return ctypes.create_string_buffer(64)


def test_quantize_validation(lib):
    ctx = ctypes.cast(_fake_ctx(), ctypes.c_void_p)
    x = ctypes.c_void_p(0x10000)
    out = ctypes.c_void_p(0x20000)

    def q(params, xp=x, rows=64, cols=64, ld=64, dt=fp4.FP4_DTYPE_BF16):
        return lib.fp4_quantize(ctx, xp, dt, rows, cols, ld, ctypes.byref(params), None, out, out, out, None)

    ok = fp4.quant_params(fp4.FP4_FMT_NVFP4)
    bad_block = fp4.quant_params(fp4.FP4_FMT_MXFP4)
    bad_block.block = 16
    assert q(bad_block) == fp4.FP4_ERR_UNSUPPORTED                     # other blocks: row-major scales only
    for blk in (48, 256, 8):
        odd = fp4.quant_params(fp4.FP4_FMT_NVFP4, sf_layout=fp4.FP4_SF_ROWMAJOR, block=blk)
        assert q(odd) == fp4.FP4_ERR_UNSUPPORTED                       # 16, 32, 64 or 128
    t64 = fp4.quant_params(fp4.FP4_FMT_NVFP4, sf_layout=fp4.FP4_SF_ROWMAJOR, transpose=True, block=64)
    assert q(t64) == fp4.FP4_ERR_UNSUPPORTED                           # row layout only
    r64 = fp4.quant_params(fp4.FP4_FMT_MXFP4, sf_layout=fp4.FP4_SF_ROWMAJOR, block=64)
    assert q(r64, cols=96, ld=96) == fp4.FP4_ERR_INVALID_ARG           # cols % 64
    assert q(r64, rows=0) == fp4.FP4_OK
    two_d_mx = fp4.quant_params(fp4.FP4_FMT_MXFP4, scaling=fp4.FP4_SCALING_2D)
    assert q(two_d_mx) == fp4.FP4_ERR_UNSUPPORTED                      # 2D scaling is NVFP4-only
    fmt7 = fp4.quant_params(fp4.FP4_FMT_NVFP4)
    fmt7.format = 7
    assert q(fmt7) == fp4.FP4_ERR_UNSUPPORTED
    assert q(ok, xp=ctypes.c_void_p(0x10008)) == fp4.FP4_ERR_MISALIGNED
    assert q(ok, ld=60, cols=60) == fp4.FP4_ERR_MISALIGNED             # pitch not 16-byte aligned
    assert q(ok, cols=40, ld=48) == fp4.FP4_ERR_INVALID_ARG            # cols % 16
    assert q(ok, ld=32) == fp4.FP4_ERR_INVALID_ARG                     # ldx < cols
    assert q(ok, dt=9) == fp4.FP4_ERR_INVALID_ARG
    assert lib.fp4_quantize(None, x, 0, 64, 64, 64, ctypes.byref(ok), None, out, out, out, None) == \
        fp4.FP4_ERR_INVALID_ARG
    assert q(ok, rows=0) == fp4.FP4_OK                                  # empty input: nothing to do


def test_gemm_validation(lib):
    ctx = ctypes.cast(_fake_ctx(), ctypes.c_void_p)
    p = 0x100000
    a = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 256, 512)
    b = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 512, 512)
    c = ctypes.c_void_p(p)
    g = lambda A, B, ldc=512: lib.fp4_gemm(ctx, ctypes.byref(A), ctypes.byref(B), fp4.FP4_DTYPE_BF16, c, ldc, 0, None)
    rm = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR, 512, 512)
    assert g(a, rm) == fp4.FP4_ERR_UNSUPPORTED                          # GEMM reads the MMA scale layout
    mx = fp4.fp4_operand(p, p, None, fp4.FP4_FMT_MXFP4, fp4.FP4_SF_MMA, 512, 512)
    assert g(a, mx) == fp4.FP4_ERR_INVALID_ARG                          # mixed formats
    k48 = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 512, 48)
    assert g(k48, k48) == fp4.FP4_ERR_INVALID_ARG                       # k % 32
    nots = fp4.fp4_operand(p, p, None, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 512, 512)
    assert g(a, nots) == fp4.FP4_ERR_INVALID_ARG                        # NVFP4 needs its tensor scale
    assert g(a, b, ldc=500) == fp4.FP4_ERR_INVALID_ARG                  # ldc < N
    assert g(a, b, ldc=516) == fp4.FP4_ERR_MISALIGNED                   # ldc * 2 % 16
    bs = fp4.fp4_operand(p, p + 4, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 512, 512)
    assert g(a, bs) == fp4.FP4_ERR_MISALIGNED                           # MMA-layout scales: 16-byte aligned
    b64 = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR, 512, 512, 64)
    assert g(a, b64) == fp4.FP4_ERR_UNSUPPORTED                         # the MMA consumes 16 / 32 only


def test_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert lib.fp4_create(ctypes.byref(h)) == fp4.FP4_ERR_CUDA


def test_hcp_num_hot_in_the_library(lib):
    """h = ceil(0.09 K) ("top 9%" of the channels) is the library's arithmetic:
    369 for K = 4096, equal to the exact rational ceiling over a range of K."""
    from fractions import Fraction
    assert lib.fp4_hcp_num_hot(4096, 0.09) == 369
    for k in list(range(0, 5000)) + [11008, 16384, 65536, 1 << 20]:
        assert lib.fp4_hcp_num_hot(k, 0.09) == -(-9 * k // 100), k
        assert lib.fp4_hcp_num_hot(k, 0.09) == int(-(-Fraction(9, 100) * k // 1))
    assert lib.fp4_hcp_num_hot(10, 1.0) == 10 and lib.fp4_hcp_num_hot(10, 0.0) == 0
    assert lib.fp4_hcp_num_hot(-1, 0.09) == -1 and lib.fp4_hcp_num_hot(10, 1.5) == -1
    assert lib.fp4_hcp_num_hot(10, float("nan")) == -1
    assert fp4.fp4_hcp_num_hot(4096) == 369


def test_hcp_select_entry_points_validate_alike(lib):
    """fp4_hcp_select and fp4_hcp_select_noalloc reject the same bad calls with
    the same status (validation runs before any CUDA call)."""
    ctx = ctypes.cast(_fake_ctx(), ctypes.c_void_p)
    p = 0x100000
    ws = ctypes.c_void_p(p)
    out = ctypes.c_void_p(p)

    def both(x, ldx, op, k_hot, hot=out):
        a = lib.fp4_hcp_select(ctx, x, ldx, ctypes.byref(op), k_hot, hot, ws, 1 << 30, None)
        b = lib.fp4_hcp_select_noalloc(x, ldx, ctypes.byref(op), k_hot, hot, None)
        return a, b

    x = ctypes.c_void_p(p)
    good = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 64, 512)
    assert both(x, 500, good, 8) == (fp4.FP4_ERR_INVALID_ARG,) * 2                # ldx < k
    assert both(ctypes.c_void_p(p + 8), 512, good, 8) == (fp4.FP4_ERR_MISALIGNED,) * 2
    assert both(x, 512, good, 513) == (fp4.FP4_ERR_INVALID_ARG,) * 2               # k_hot > k
    assert both(x, 512, good, 8, None) == (fp4.FP4_ERR_INVALID_ARG,) * 2           # no output
    b64 = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR, 64, 512, 64)
    assert both(x, 512, b64, 8) == (fp4.FP4_ERR_UNSUPPORTED,) * 2
    nots = fp4.fp4_operand(p, p, None, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 64, 512)
    assert both(x, 512, nots, 8) == (fp4.FP4_ERR_INVALID_ARG,) * 2                 # NVFP4 tensor scale
    # an empty input with an unaligned pointer is accepted by both (nothing is read)
    empty = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA, 0, 512)
    assert both(ctypes.c_void_p(p + 8), 512, empty, 0) == (fp4.FP4_OK,) * 2
    wide = fp4.fp4_operand(p, p, p, fp4.FP4_FMT_MXFP4, fp4.FP4_SF_MMA, 16, fp4.FP4_NOALLOC_MAX_CHANNELS + 32)
    assert lib.fp4_hcp_select_noalloc(x, fp4.FP4_NOALLOC_MAX_CHANNELS + 32, ctypes.byref(wide), 8, out,
                                      None) == fp4.FP4_ERR_TOO_LARGE
