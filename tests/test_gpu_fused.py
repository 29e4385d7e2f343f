"""The GEMM with the activation's quantization fused into its operand producer
(fp4_gemm_quant_a): MXFP4, round to nearest, 1D blocks of 32 along K, the
forward operand of the outlier page's recipe (§4.1), formed from bf16 X inside
the CTA-pair GEMM.

Checks, through the C ABI:
  * the codes and scales the kernel writes out equal the oracle's quantization
    of X byte for byte (and fp4_quantize's, padding included);
  * the product equals fp4_quantize + fp4_gemm bit for bit (same tiles, same
    MMA order), and the oracle's GEMM of the oracle's codes within the GEMM
    bound (|Y - Y_ref| <= 1e-3 sum |a||b|, + 2^-8 |Y_ref| for bf16 output);
  * ragged M, N and K (K not a multiple of the 256-element stage), more tiles
    than CTA pairs, bf16 and fp32 output, rows of X with a pitch;
  * the argument checks.
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o
from _util import mismatch_report, untile_scales

pytestmark = pytest.mark.gpu

MX = fp4.FP4_FMT_MXFP4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    from fp4_block_scaled_e8m0_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    fp4.load_library()


def _x(rng, M, K, pitch=0):
    """Student-t(3) activations with 1% hot channels x100, bf16, optional row pitch."""
    x = rng.standard_t(3, (M, K)).astype(np.float32)
    x[:, rng.permutation(K)[: max(1, K // 100)]] *= 100
    full = np.zeros((M, K + pitch), np.float32)
    full[:, :K] = x
    t = torch.from_numpy(full).to(torch.bfloat16).cuda()
    return t[:, :K], t[:, :K].float().cpu().numpy()


def _w(rng, N, K):
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    t = torch.from_numpy(w).to(torch.bfloat16)
    return t.cuda(), t.float().numpy()


def _fused_and_unfused(x, wq, out_dtype):
    M, K = x.shape
    a_out = fp4.alloc_qtensor(M, K, MX, fp4.FP4_SF_MMA, x.device)
    a_out.scales.fill_(0xAB)        # every byte, padding included, must be written
    y = fp4.fp4_gemm_quant_a(x, wq, out_dtype=out_dtype, a_out=a_out)
    xq = fp4.fp4_quantize(x, fp4.quant_params(MX))
    y_ref = fp4.fp4_gemm(xq, wq, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y, a_out, y_ref, xq


@pytest.mark.parametrize("M,N,K,out_dtype,pitch", [
    (256, 256, 256, torch.bfloat16, 0),
    (300, 520, 800, torch.bfloat16, 8),      # ragged M, N and a K tail inside the last stage
    (129, 264, 4096, torch.float32, 0),      # 16 K stages, one row past a 128-row tile
    (520, 776, 1056, torch.float32, 24),
])
def test_fused_matches_oracle_and_unfused(M, N, K, out_dtype, pitch):
    rng = np.random.default_rng(1000 + M + N + K)
    x, xn = _x(rng, M, K, pitch)
    w, wn = _w(rng, N, K)
    wq = fp4.fp4_quantize(w, fp4.quant_params(MX))
    y, a_out, y_ref, xq = _fused_and_unfused(x, wq, out_dtype)
    # the quantization written out: the oracle's bytes, and fp4_quantize's (padding too)
    ca, sa, _ = o.quantize(xn, o.MXFP4)
    got_c = a_out.codes.cpu().numpy()
    got_s = untile_scales(a_out.scales.cpu().numpy(), M, K // 32)
    assert np.array_equal(got_s, sa), mismatch_report(got_s, sa, "scales vs oracle")
    assert np.array_equal(got_c, ca), mismatch_report(got_c, ca, "codes vs oracle")
    assert torch.equal(a_out.scales, xq.scales), "scale buffer differs from fp4_quantize's"
    # the product: bit-identical to quantize-then-GEMM, within the bound of the oracle's
    assert torch.equal(y.view(torch.int16) if out_dtype == torch.bfloat16 else y.view(torch.int32),
                       y_ref.view(torch.int16) if out_dtype == torch.bfloat16 else y_ref.view(torch.int32)), \
        "fused GEMM differs from fp4_quantize + fp4_gemm"
    cb, sb, _ = o.quantize(wn, o.MXFP4)
    yo, bound = o.gemm(ca, sa, cb, sb, o.MXFP4, None, None)
    got = y.float().cpu().numpy().astype(np.float64)
    tol = o.gemm_tolerance(bound, yo, out_dtype == torch.bfloat16) + 1e-30
    bad = np.abs(got - yo) > tol
    assert not bad.any(), f"{bad.sum()} elements outside the GEMM bound"


def test_fused_many_tiles_bit_identical():
    """More 256 x 256 tiles (9 x 33) than CTA pairs, ragged in both dimensions;
    every element against the unfused path, the codes against fp4_quantize."""
    rng = np.random.default_rng(7)
    M, N, K = 2200, 8392, 512
    x, _ = _x(rng, M, K)
    w, _ = _w(rng, N, K)
    wq = fp4.fp4_quantize(w, fp4.quant_params(MX))
    y, a_out, y_ref, xq = _fused_and_unfused(x, wq, torch.bfloat16)
    assert torch.equal(a_out.codes, xq.codes) and torch.equal(a_out.scales, xq.scales)
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_fused_without_quantized_output():
    rng = np.random.default_rng(8)
    x, _ = _x(rng, 384, 1024)
    w, _ = _w(rng, 512, 1024)
    wq = fp4.fp4_quantize(w, fp4.quant_params(MX))
    y = fp4.fp4_gemm_quant_a(x, wq)
    y_ref = fp4.fp4_gemm(fp4.fp4_quantize(x, fp4.quant_params(MX)), wq)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_fused_argument_checks():
    lib = fp4.load_library()
    import ctypes
    x = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((64, 64), dtype=torch.bfloat16, device="cuda")

    def call(xt, bq, ldx=256, codes=None, scales=None, ldc=64):
        ob = bq.operand()
        return lib.fp4_gemm_quant_a(fp4._ctx(None), ctypes.c_void_p(xt.data_ptr()), xt.shape[0], ldx, ctypes.byref(ob),
                                    fp4.FP4_DTYPE_BF16, ctypes.c_void_p(y.data_ptr()), ldc,
                                    None if codes is None else ctypes.c_void_p(codes.data_ptr()),
                                    None if scales is None else ctypes.c_void_p(scales.data_ptr()), None)

    wq_mx = fp4.fp4_quantize(w, fp4.quant_params(MX))
    wq_nv = fp4.fp4_quantize(w, fp4.quant_params(fp4.FP4_FMT_NVFP4))
    wq_rm = fp4.fp4_quantize(w, fp4.quant_params(MX, sf_layout=fp4.FP4_SF_ROWMAJOR))
    codes = torch.empty((64, 128), dtype=torch.uint8, device="cuda")
    assert call(x, wq_nv) == fp4.FP4_ERR_UNSUPPORTED
    assert call(x, wq_rm) == fp4.FP4_ERR_UNSUPPORTED
    assert call(x, wq_mx, codes=codes) == fp4.FP4_ERR_INVALID_ARG          # codes without scales
    assert call(x, wq_mx, ldx=260) == fp4.FP4_ERR_MISALIGNED               # pitch not 16 bytes
    assert call(x, wq_mx, ldx=200) == fp4.FP4_ERR_INVALID_ARG              # pitch < k
    assert call(x, wq_mx, ldc=32) == fp4.FP4_ERR_INVALID_ARG               # ldc < N
    assert call(x, wq_mx) == fp4.FP4_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,N,K", [(1, 256, 256), (200, 8, 32), (130, 264, 96)])
def test_fused_edge_shapes(M, N, K):
    """One row; eight output columns and K = 32 (one block, a stage mostly
    zero-filled); K not a multiple of 128: equal to fp4_quantize + fp4_gemm and
    to the oracle's codes."""
    rng = np.random.default_rng(M * 7 + N + K)
    x, xn = _x(rng, M, K)
    w, _ = _w(rng, N, K)
    wq = fp4.fp4_quantize(w, fp4.quant_params(MX))
    y, a_out, y_ref, xq = _fused_and_unfused(x, wq, torch.float32)
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
    ca, sa, _ = o.quantize(xn, o.MXFP4)
    assert np.array_equal(a_out.codes.cpu().numpy(), ca)
    assert np.array_equal(untile_scales(a_out.scales.cpu().numpy(), M, K // 32), sa)


def test_fused_empty_operands():
    """No rows of X, or no rows of B: nothing to compute, FP4_OK."""
    w, _ = _w(np.random.default_rng(1), 64, 256)
    wq = fp4.fp4_quantize(w, fp4.quant_params(MX))
    x0 = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    assert fp4.fp4_gemm_quant_a(x0, wq).shape == (0, 64)
    x, _ = _x(np.random.default_rng(2), 32, 256)
    w0 = fp4.fp4_quantize(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"), fp4.quant_params(MX))
    assert fp4.fp4_gemm_quant_a(x, w0).shape == (32, 0)
    torch.cuda.synchronize()
    assert fp4.fp4_sync_status() == fp4.FP4_OK
