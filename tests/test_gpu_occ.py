"""GPU <-> oracle parity for outlier clamping and compensation (OCC, the MSR
write-up §三 and §六) and the quantization-quality statistics, through the C ABI.

Bit-exact: the threshold tau and the outlier count (integer selection), the
codes, scales and tensor scale of the clamped quantization, the per-column
outlier counts.  The OCC GEMM within the FP4 GEMM bound plus the rounding the
compensation adds: the dense columns carry bf16(dX / alpha) (<= 2^-9 relative
each, plus the fp32 rounding of 1/alpha), so 2^-8 sum |dX||W| more; the
scattered outliers are added in the GEMM epilogue, and a bf16 output is
rounded before and after that addition: 2^-9 (|Y - S| + |Y|) <= 2^-8 (|Y| +
sum |dX||W|) with S the scattered part.  The fp64 sums of the statistics within
1e-9 relative (summation order only).
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o
from _util import mismatch_report, untile_scales
from fp4_block_scaled_e8m0_gb300 import inputs

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


def _hot_t(rows, cols, seed, dtype=torch.bfloat16):
    rng = np.random.default_rng(seed)
    x = rng.standard_t(3, (rows, cols)).astype(np.float32)
    hot = rng.permutation(cols)[: max(1, cols // 100)]
    x[:, hot] *= 100
    t = torch.from_numpy(x).to(dtype)
    return t, t.float().numpy()


def _gpu_quant_np(q):
    codes = q.codes.cpu().numpy()
    nsf = q.k // fp4.BLOCK[q.fmt]
    sc = q.scales.cpu().numpy()
    scales = untile_scales(sc, q.rows, nsf) if q.sf_layout == fp4.FP4_SF_MMA else sc[: q.rows * nsf].reshape(q.rows, nsf)
    g = q.tensor_scale.cpu().numpy()[0] if q.tensor_scale is not None else None
    return codes, scales, g


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("q", [0.5, 0.99, 0.999, 1.0])
def test_threshold_exact(dtype, q):
    for shape, seed in (((333, 320), 40), ((64, 8), 41)):
        x, xn = _hot_t(*shape, seed, dtype)
        if seed == 41:
            xn = np.round(xn * 2) / 2                      # many ties
            x = torch.from_numpy(xn).to(dtype)
            xn = x.float().numpy()
        tau, n_out = fp4.fp4_occ_threshold(x.cuda(), q)
        want = o.occ_threshold(xn, q)
        got = tau.cpu().numpy()[0]
        assert got.view(np.uint32) == np.float32(want).view(np.uint32), (got, want)
        assert int(n_out.cpu()[0]) == int(np.count_nonzero(np.abs(xn) > want))


def test_threshold_pitched_and_empty():
    x, xn = _hot_t(100, 128, 42)
    buf = torch.zeros((100, 160), dtype=torch.bfloat16, device="cuda")
    buf[:, :128] = x.cuda()
    buf[:, 128:] = 1e4                                      # the pitch gap must be ignored
    tau, n_out = fp4.fp4_occ_threshold(buf[:, :128])
    assert tau.item() == float(o.occ_threshold(xn))
    assert n_out.item() == int(np.count_nonzero(np.abs(xn) > o.occ_threshold(xn)))
    tau, n_out = fp4.fp4_occ_threshold(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"))
    assert tau.item() == 0.0 and n_out.item() == 0


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_occ_quantize_bit_exact(fmt, sf_layout, rounding):
    x, xn = _hot_t(333, 320, 43)
    tau, _ = fp4.fp4_occ_threshold(x.cuda())
    counts = torch.empty((320,), dtype=torch.float32, device="cuda")
    rnd = fp4.FP4_ROUND_SR if rounding == "sr" else fp4.FP4_ROUND_RTN
    p = fp4.quant_params(fmt, rnd, sf_layout=sf_layout, sr_seed=7, sr_stream=1, sr_offset=3)
    q = fp4.fp4_occ_quantize(x.cuda(), p, tau, col_counts=counts)
    t = o.occ_threshold(xn)
    xc, _ = o.occ_split(xn, t)
    wc, ws, wg = o.quantize(xc, FMT[fmt], rounding, sr_seed=7, sr_stream=1, sr_offset=3)
    codes, scales, g = _gpu_quant_np(q)
    assert np.array_equal(scales, ws), mismatch_report(scales, ws, "scales")
    assert np.array_equal(codes, wc), mismatch_report(codes, wc, "codes")
    if wg is not None:
        assert np.float32(g).view(np.uint32) == np.float32(wg).view(np.uint32)
    assert np.array_equal(counts.cpu().numpy(), (np.abs(xn) > t).sum(axis=0).astype(np.float32))


def test_occ_quantize_rejects_transpose_and_rht():
    x, _ = _hot_t(64, 64, 44)
    tau, _ = fp4.fp4_occ_threshold(x.cuda())
    for p in (fp4.quant_params(transpose=True), fp4.quant_params(rht=True)):
        with pytest.raises(fp4.FP4Error):
            fp4.fp4_occ_quantize(x.cuda(), p, tau)


def occ_gemm_tolerance(xn, wn, tau, y_ref, bound, out_bf16):
    _, dx = o.occ_split(xn, tau)
    comp = np.abs(dx.astype(np.float64)) @ np.abs(wn.astype(np.float64)).T
    tol = 1e-3 * bound + 2.0 ** -8 * comp
    if out_bf16:
        tol = tol + 2.0 ** -8 * (np.abs(y_ref) + comp)
    return tol


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("k_dense", [0, 3, 64])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_occ_gemm(fmt, k_dense, out_dtype):
    M, K, N = 300, 512, 264
    x, xn = _hot_t(M, K, 45)
    rng = np.random.default_rng(46)
    w = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    wn = w.float().numpy()
    xd, wd = x.cuda(), w.cuda()
    tau, _ = fp4.fp4_occ_threshold(xd)
    counts = torch.empty((K,), dtype=torch.float32, device="cuda")
    xq = fp4.fp4_occ_quantize(xd, fp4.quant_params(fmt), tau, col_counts=counts)
    wq = fp4.fp4_quantize(wd, fp4.quant_params(fmt))
    y = fp4.fp4_occ_gemm(xd, wd, xq, wq, tau, counts, k_dense, fp4.fp4_occ_max_outliers(M, K), out_dtype)
    assert fp4.fp4_sync_status() == 0
    t = o.occ_threshold(xn)
    y_ref, bound, _, _ = o.occ_gemm(xn, wn, FMT[fmt], t)
    got = y.float().cpu().numpy().astype(np.float64)
    tol = occ_gemm_tolerance(xn, wn, t, y_ref, bound, out_dtype == torch.bfloat16)
    err = np.abs(got - y_ref)
    assert np.all(err <= tol), f"{(err > tol).sum()} off; worst {np.max(err / tol)} of the tolerance"
    # the compensation is real: without it most outputs fall outside the tolerance
    xq_y = fp4.fp4_gemm(xq, wq, out_dtype=torch.float32).cpu().numpy()
    assert (np.abs(xq_y - y_ref) > tol).mean() > 0.5


def test_occ_gemm_fp32_x_ragged_n():
    M, K, N = 200, 256, 100                 # N not a multiple of 8: pitched output
    x, xn = _hot_t(M, K, 47, torch.float32)
    rng = np.random.default_rng(48)
    w = torch.from_numpy((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    wn = w.float().numpy()
    xd, wd = x.cuda(), w.cuda()
    tau, _ = fp4.fp4_occ_threshold(xd)
    counts = torch.empty((K,), dtype=torch.float32, device="cuda")
    xq = fp4.fp4_occ_quantize(xd, fp4.quant_params(fp4.FP4_FMT_NVFP4), tau, col_counts=counts)
    wq = fp4.fp4_quantize(wd, fp4.quant_params(fp4.FP4_FMT_NVFP4))
    buf = torch.full((M, 104), 5.0, dtype=torch.bfloat16, device="cuda")
    fp4.fp4_occ_gemm(xd, wd, xq, wq, tau, counts, 2, fp4.fp4_occ_max_outliers(M, K), out=buf[:, :N])
    t = o.occ_threshold(xn)
    y_ref, bound, _, _ = o.occ_gemm(xn, wn, o.NVFP4, t)
    got = buf[:, :N].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - y_ref) <= occ_gemm_tolerance(xn, wn, t, y_ref, bound, True))
    assert torch.all(buf[:, N:] == 5.0)


def test_occ_gemm_capacity_overflow_sets_status():
    # a scattered list larger than max_outliers: the rows that do not fit are
    # left out and the context reports FP4_ERR_TOO_LARGE (no fault)
    M, K, N = 128, 256, 64
    x, _ = _hot_t(M, K, 49)
    w = torch.ones((N, K), dtype=torch.bfloat16, device="cuda")
    xd = x.cuda()
    tau, _ = fp4.fp4_occ_threshold(xd)
    xq = fp4.fp4_occ_quantize(xd, fp4.quant_params(fp4.FP4_FMT_NVFP4), tau)
    wq = fp4.fp4_quantize(w, fp4.quant_params(fp4.FP4_FMT_NVFP4))
    fp4.fp4_occ_gemm(xd, w, xq, wq, tau, None, 0, 1)
    assert fp4.fp4_sync_status() == fp4.FP4_ERR_TOO_LARGE
    assert fp4.fp4_sync_status() == 0                       # read and cleared


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
def test_quant_error_stats(fmt, sf_layout):
    x, xn = _hot_t(333, 320, 50)
    xd = x.cuda()
    q_direct = fp4.fp4_quantize(xd, fp4.quant_params(fmt, sf_layout=sf_layout))
    tau, _ = fp4.fp4_occ_threshold(xd)
    q_occ = fp4.fp4_occ_quantize(xd, fp4.quant_params(fmt, sf_layout=sf_layout), tau)
    s_direct, st_direct = (t.cpu().numpy() for t in fp4.fp4_quant_error_stats(xd, q_direct))
    s_occ, st_occ = (t.cpu().numpy() for t in fp4.fp4_quant_error_stats(xd, q_occ, tau))
    c, s, g = o.quantize(xn, FMT[fmt])
    h_direct = o.dequantize(c, s, FMT[fmt], g).astype(np.float64)
    h_occ = o.occ_reconstruction(xn, FMT[fmt], o.occ_threshold(xn))
    for got, hat in ((s_direct, h_direct), (s_occ, h_occ)):
        a = xn.astype(np.float64).reshape(-1)
        b = hat.reshape(-1)
        want = np.array([a @ a, b @ b, a @ b, ((a - b) ** 2).sum()])
        assert np.allclose(got, want, rtol=1e-9, atol=0), (got, want)
    # the library's cosine / MSE / SNR / relative error against the oracle's
    for st, hat in ((st_direct, h_direct), (st_occ, h_occ)):
        got = fp4.stats_dict(st)
        ref = o.quant_error_stats(xn, hat)
        assert abs(got["cos"] - ref["cos"]) < 1e-9 and abs(got["snr_db"] - ref["snr_db"]) < 1e-6
        assert abs(got["mse"] - ref["mse"]) <= 1e-9 * ref["mse"]
        assert abs(got["rel_err"] - o.relative_error(xn, hat)) <= 1e-9 * o.relative_error(xn, hat)
    st_d, st_o = fp4.stats_dict(st_direct), fp4.stats_dict(st_occ)
    assert st_o["snr_db"] > st_d["snr_db"] and st_o["cos"] > st_d["cos"]
