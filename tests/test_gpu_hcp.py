"""GPU <-> oracle parity for hot-channel compensation, through the C ABI.

Selection: the set of k_hot channels must equal the oracle's, except for
channels whose error lies within 1e-5 (relative) of the k-th largest error
(the GPU sums the per-channel errors in fp32 in a different order).  The
planted x100 channels must be selected.
GEMM (single- and two-kernel modes, orders 1 and 2): the GEMM bound with the
oracle's bf16 residual columns.
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o

pytestmark = pytest.mark.gpu

FMT = {fp4.FP4_FMT_MXFP4: o.MXFP4, fp4.FP4_FMT_NVFP4: o.NVFP4}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    from fp4_block_scaled_e8m0_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    fp4.load_library()


def _data(fmt, M=320, K=512, N=264, seed=1):
    rng = np.random.default_rng(seed)
    x = rng.standard_t(3, (M, K)).astype(np.float32)
    hot = np.sort(rng.permutation(K)[: max(1, K // 100)])
    x[:, hot] *= 100
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    return xt, wt, xt.float().numpy(), wt.float().numpy(), hot


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
def test_hcp_select_matches_oracle(fmt):
    xt, _, xn, _, planted = _data(fmt)
    K = xn.shape[1]
    h = fp4.fp4_hcp_num_hot(K)
    xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fmt))
    got = fp4.fp4_hcp_select(xt.cuda(), xq, h).cpu().numpy()
    assert np.all(np.diff(got) > 0), "indices must be ascending and distinct"
    c, s, g = o.quantize(xn, FMT[fmt])
    e = o.hcp_channel_errors(xn, c, s, FMT[fmt], g)
    want = o.hcp_select(xn, c, s, FMT[fmt], g, h)
    kth = np.sort(e)[::-1][h - 1]
    band = np.abs(e - kth) <= 1e-5 * kth
    diff = set(got.tolist()) ^ set(want.tolist())
    assert all(band[i] for i in diff), f"selection differs outside the tie band: {sorted(diff)[:10]}"
    assert set(planted.tolist()) <= set(got.tolist())


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("mode", [fp4.FP4_HCP_SINGLE, fp4.FP4_HCP_TWO])
@pytest.mark.parametrize("order", [1, 2])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_hcp_gemm_matches_oracle(fmt, mode, order, out_dtype):
    xt, wt, xn, wn, _ = _data(fmt, seed=2)
    K = xn.shape[1]
    h = fp4.fp4_hcp_num_hot(K)
    xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fmt))
    wq = fp4.fp4_quantize(wt.cuda(), fp4.quant_params(fmt))
    cx, sx, gx = o.quantize(xn, FMT[fmt])
    cw, sw, gw = o.quantize(wn, FMT[fmt])
    hot = o.hcp_select(xn, cx, sx, FMT[fmt], gx, h)
    y = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, torch.from_numpy(hot).cuda(), h, mode, order, out_dtype)
    got = y.float().cpu().numpy().astype(np.float64)
    yref, bound = o.hcp_gemm(xn, cx, sx, wn, cw, sw, FMT[fmt], gx, gw, hot, order)
    tol = o.gemm_tolerance(bound, yref, out_dtype == torch.bfloat16)
    if mode == fp4.FP4_HCP_TWO and out_dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * np.abs(yref)          # the base result is rounded to bf16 once more
    err = np.abs(got - yref)
    assert np.all(err <= tol), f"{(err > tol).sum()} outside; worst {np.max(err - tol)}"


def test_hcp_zero_hot_is_plain_gemm():
    xt, wt, xn, wn, _ = _data(fp4.FP4_FMT_NVFP4, seed=3)
    xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fp4.FP4_FMT_NVFP4))
    wq = fp4.fp4_quantize(wt.cuda(), fp4.quant_params(fp4.FP4_FMT_NVFP4))
    y0 = fp4.fp4_gemm(xq, wq, torch.float32)
    y1 = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, torch.zeros(1, dtype=torch.int32, device="cuda"), 0,
                          out_dtype=torch.float32)
    assert torch.equal(y0, y1)


def _quant_np(q):
    from _util import untile_scales
    codes = q.codes.cpu().numpy()
    nsf = q.k // fp4.BLOCK[q.fmt]
    sc = q.scales.cpu().numpy()
    scales = untile_scales(sc, q.rows, nsf) if q.sf_layout == fp4.FP4_SF_MMA else sc[: q.rows * nsf].reshape(q.rows, nsf)
    g = q.tensor_scale.cpu().numpy()[0] if q.tensor_scale is not None else None
    return codes, scales, g


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
@pytest.mark.parametrize("rounding", [fp4.FP4_ROUND_RTN, fp4.FP4_ROUND_SR])
def test_hcp_quantize_zeroed_bit_exact(fmt, sf_layout, rounding):
    xt, _, xn, _, planted = _data(fmt, M=333, K=512, seed=4)
    hot = np.sort(np.concatenate([planted, [0, 1, 2, 511]]))   # edges of the row too
    p = fp4.quant_params(fmt, rounding, sf_layout=sf_layout, sr_seed=3, sr_stream=1)
    q = fp4.fp4_hcp_quantize_zeroed(xt.cuda(), p, torch.from_numpy(hot.astype(np.int32)).cuda(), len(hot))
    wc, ws, wg = o.quantize(o.hcp_zero_columns(xn, hot), FMT[fmt], "sr" if rounding else "rtn", sr_seed=3,
                            sr_stream=1)
    codes, scales, g = _quant_np(q)
    assert np.array_equal(scales, ws)
    assert np.array_equal(codes, wc)
    if wg is not None:
        assert np.float32(g).view(np.uint32) == np.float32(wg).view(np.uint32)


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("mode", [fp4.FP4_HCP_SINGLE, fp4.FP4_HCP_TWO])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_hcp_zeroed_gemm_matches_oracle(fmt, mode, out_dtype):
    xt, wt, xn, wn, _ = _data(fmt, seed=5)
    K = xn.shape[1]
    h = fp4.fp4_hcp_num_hot(K)
    cx, sx, gx = o.quantize(xn, FMT[fmt])
    hot = o.hcp_select(xn, cx, sx, FMT[fmt], gx, h)
    hot_d = torch.from_numpy(hot.astype(np.int32)).cuda()
    x0q = fp4.fp4_hcp_quantize_zeroed(xt.cuda(), fp4.quant_params(fmt), hot_d, h)
    wq = fp4.fp4_quantize(wt.cuda(), fp4.quant_params(fmt))
    y = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), x0q, wq, hot_d, h, mode, 0, out_dtype)
    got = y.float().cpu().numpy().astype(np.float64)
    yref, bound, _, _ = o.hcp_zeroed_gemm(xn, wn, FMT[fmt], hot)
    tol = o.gemm_tolerance(bound, yref, out_dtype == torch.bfloat16)
    if mode == fp4.FP4_HCP_TWO and out_dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * np.abs(yref)
    err = np.abs(got - yref)
    assert np.all(err <= tol), f"{(err > tol).sum()} outside; worst {np.max(err - tol)}"
    # closer to the unquantized product than the order-2 compensation on these activations
    exact = xn.astype(np.float64) @ wn.astype(np.float64).T
    xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fmt))
    y2 = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, hot_d, h, mode, 2, torch.float32).cpu().numpy()
    assert np.abs(got - exact).sum() < np.abs(y2 - exact).sum() * 1.5


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("order", [0, 1, 2])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_hcp_fp8_tail_matches_oracle(fmt, order, out_dtype):
    # E4M3 extra columns (tcgen05 kind::f8f6f4) with per-row scales, added by a
    # second GEMM; the oracle uses the same E4M3 values, so the GEMM bound holds
    xt, wt, xn, wn, _ = _data(fmt, seed=6)
    K = xn.shape[1]
    h = fp4.fp4_hcp_num_hot(K)
    cx, sx, gx = o.quantize(xn, FMT[fmt])
    hot = o.hcp_select(xn, cx, sx, FMT[fmt], gx, h)
    hot_d = torch.from_numpy(hot.astype(np.int32)).cuda()
    if order == 0:
        xq = fp4.fp4_hcp_quantize_zeroed(xt.cuda(), fp4.quant_params(fmt), hot_d, h)
        cx, sx, gx = o.quantize(o.hcp_zero_columns(xn, hot), FMT[fmt])
    else:
        xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fmt))
    wq = fp4.fp4_quantize(wt.cuda(), fp4.quant_params(fmt))
    cw, sw, gw = o.quantize(wn, FMT[fmt])
    y = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, hot_d, h, fp4.FP4_HCP_TWO_FP8, order, out_dtype)
    got = y.float().cpu().numpy().astype(np.float64)
    yref, bound = o.hcp_gemm_fp8(xn, cx, sx, wn, cw, sw, FMT[fmt], gx, gw, hot, order)
    tol = o.gemm_tolerance(bound, yref, out_dtype == torch.bfloat16)
    if out_dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * np.abs(yref)          # the base result is rounded to bf16 once more
    err = np.abs(got - yref)
    assert np.all(err <= tol), f"{(err > tol).sum()} outside; worst {np.max(err - tol)}"
    # the FP8 tail does compensate: closer to the unquantized product than plain FP4
    exact = xn.astype(np.float64) @ wn.astype(np.float64).T
    y0 = fp4.fp4_gemm(xq, wq, torch.float32).cpu().numpy()
    assert np.abs(got - exact).sum() < np.abs(y0 - exact).sum()


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("order", [0, 1, 2])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(320, 512, 264, 6), (700, 1024, 520, 7)])
def test_hcp_mxfp8_single_kernel_matches_oracle(fmt, order, out_dtype, shape):
    # MXFP8 extra columns (E4M3, E8M0 per 32; tcgen05 kind::mxf8f6f4) in the FP4
    # accumulator of one CTA-pair kernel; the oracle uses the same MXFP8 values,
    # so the GEMM bound holds.  The second shape has several 256 x 256 tiles,
    # ragged edges and more hot channels than one 128-column stage holds.
    M, K, N, seed = shape
    xt, wt, xn, wn, _ = _data(fmt, M=M, K=K, N=N, seed=seed)
    h = fp4.fp4_hcp_num_hot(K)
    cx, sx, gx = o.quantize(xn, FMT[fmt])
    hot = o.hcp_select(xn, cx, sx, FMT[fmt], gx, h)
    hot_d = torch.from_numpy(hot.astype(np.int32)).cuda()
    if order == 0:
        xq = fp4.fp4_hcp_quantize_zeroed(xt.cuda(), fp4.quant_params(fmt), hot_d, h)
        cx, sx, gx = o.quantize(o.hcp_zero_columns(xn, hot), FMT[fmt])
    else:
        xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fmt))
    wq = fp4.fp4_quantize(wt.cuda(), fp4.quant_params(fmt))
    cw, sw, gw = o.quantize(wn, FMT[fmt])
    y = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, hot_d, h, fp4.FP4_HCP_SINGLE_MXFP8, order, out_dtype)
    got = y.float().cpu().numpy().astype(np.float64)
    yref, bound = o.hcp_gemm_mxfp8(xn, cx, sx, wn, cw, sw, FMT[fmt], gx, gw, hot, order)
    tol = o.gemm_tolerance(bound, yref, out_dtype == torch.bfloat16)
    err = np.abs(got - yref)
    assert np.all(err <= tol), f"{(err > tol).sum()} outside; worst {np.max(err - tol)}"
    assert fp4.fp4_sync_status() == fp4.FP4_OK
    # and it compensates: closer to the unquantized product than the plain FP4 GEMM
    exact = xn.astype(np.float64) @ wn.astype(np.float64).T
    y0 = fp4.fp4_gemm(xq, wq, torch.float32).cpu().numpy()
    assert np.abs(got - exact).sum() < np.abs(y0 - exact).sum()


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
def test_hcp_mxfp8_hot_list_in_any_order(fmt):
    # the extra columns follow the order of hot_idx, ascending or not
    xt, wt, xn, wn, _ = _data(fmt, M=300, K=1024, N=264, seed=9)
    h = fp4.fp4_hcp_num_hot(1024)
    cx, sx, gx = o.quantize(xn, FMT[fmt])
    hot = np.random.default_rng(3).permutation(o.hcp_select(xn, cx, sx, FMT[fmt], gx, h))
    hot_d = torch.from_numpy(hot.astype(np.int32)).cuda()
    xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fmt))
    wq = fp4.fp4_quantize(wt.cuda(), fp4.quant_params(fmt))
    cw, sw, gw = o.quantize(wn, FMT[fmt])
    y = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, hot_d, h, fp4.FP4_HCP_SINGLE_MXFP8, 2, torch.float32)
    yref, bound = o.hcp_gemm_mxfp8(xn, cx, sx, wn, cw, sw, FMT[fmt], gx, gw, hot, 2)
    err = np.abs(y.cpu().numpy().astype(np.float64) - yref)
    assert np.all(err <= o.gemm_tolerance(bound, yref, False))


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("order", [0, 2])
def test_hcp_wide_rows_take_the_per_element_gathers(fmt, order):
    # K = 20480: a row's two staging buffers no longer fit the shared-memory
    # budget, so both gathers (bf16 and MXFP8 columns) read the hot values
    # directly; same oracle products as at small K
    M, K, N = 130, 20480, 136
    xt, wt, xn, wn, _ = _data(fmt, M=M, K=K, N=N, seed=21)
    h = fp4.fp4_hcp_num_hot(K)
    cx, sx, gx = o.quantize(xn, FMT[fmt])
    hot = o.hcp_select(xn, cx, sx, FMT[fmt], gx, h)
    hot_d = torch.from_numpy(hot.astype(np.int32)).cuda()
    if order == 0:
        xq = fp4.fp4_hcp_quantize_zeroed(xt.cuda(), fp4.quant_params(fmt), hot_d, h)
        cx, sx, gx = o.quantize(o.hcp_zero_columns(xn, hot), FMT[fmt])
    else:
        xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fmt))
    wq = fp4.fp4_quantize(wt.cuda(), fp4.quant_params(fmt))
    cw, sw, gw = o.quantize(wn, FMT[fmt])
    y = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, hot_d, h, fp4.FP4_HCP_SINGLE, order, torch.float32)
    if order == 0:
        yref, bound, _, _ = o.hcp_zeroed_gemm(xn, wn, FMT[fmt], hot)
    else:
        yref, bound = o.hcp_gemm(xn, cx, sx, wn, cw, sw, FMT[fmt], gx, gw, hot, order)
    err = np.abs(y.cpu().numpy().astype(np.float64) - yref)
    assert np.all(err <= o.gemm_tolerance(bound, yref, False)), "bf16 columns"
    y8 = fp4.fp4_hcp_gemm(xt.cuda(), wt.cuda(), xq, wq, hot_d, h, fp4.FP4_HCP_SINGLE_MXFP8, order, torch.float32)
    yref8, bound8 = o.hcp_gemm_mxfp8(xn, cx, sx, wn, cw, sw, FMT[fmt], gx, gw, hot, order)
    err8 = np.abs(y8.cpu().numpy().astype(np.float64) - yref8)
    assert np.all(err8 <= o.gemm_tolerance(bound8, yref8, False)), "MXFP8 columns"
    assert fp4.fp4_sync_status() == fp4.FP4_OK
