"""Parity at the benchmark workloads' full sizes, in the launch configuration the
benchmark times.  Quantized tensors are checked bit for bit on sampled row
blocks (the oracle quantizes those rows with the tensor's full amax); GEMM
outputs on sampled rows (all columns), computed by the oracle one row at a time.

Workloads: the small linear fprop (X 256x512, W 512x512, MXFP4), the NVFP4
4096x4096 tensor with outlier columns (RTN, SR, DGE), the LLaMA-1B MLP
up-projection fwd+bwd (NVFP4, SR + RHT + 2D backward), the 7B FFN GEMMs in MXFP4
and the hot-channel-compensated NVFP4 GEMM.
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o
from _util import mismatch_report, untile_scales

pytestmark = pytest.mark.gpu
NV, MX = fp4.FP4_FMT_NVFP4, fp4.FP4_FMT_MXFP4
OF = {MX: o.MXFP4, NV: o.NVFP4}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    from fp4_block_scaled_e8m0_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    fp4.load_library()


def _sample_rows(n, count, seed):
    rng = np.random.default_rng(seed)
    idx = np.concatenate([[0, n - 1], rng.choice(n, size=min(count, n), replace=False)])
    return np.unique(idx)


def _oracle_rows(x_np, fmt_gpu, params_oracle, rows_out):
    """The oracle's quantization of output rows `rows_out` (the output layout's
    rows; for a transposed output these are input columns), from the input
    values alone.  NVFP4 takes the full tensor's amax (after any RHT).  For 2D
    scaling the rows are widened to whole 16-row groups.  Returns (codes,
    scales, g, rows)."""
    fmt = OF[fmt_gpu]
    transpose = params_oracle.get("transpose", False)
    rht = params_oracle.get("rht", False)
    w = x_np.T if transpose else x_np
    given = None
    if fmt_gpu == NV:
        ww = o.rht16(np.ascontiguousarray(w), 1, params_oracle.get("rht_seed", 0)) if rht else w
        given = o.tensor_amax(ww)
    two_d = params_oracle.get("scaling") == "2d"
    rows_out = np.unique(np.asarray(rows_out))
    if two_d:
        rows_out = np.unique(np.concatenate([np.arange(r - r % 16, r - r % 16 + 16) for r in rows_out]))
    kw = {k: v for k, v in params_oracle.items() if k not in ("transpose",)}
    # the SR counter of output element (r, c) is r * cols + c: a slice starting
    # at row r0 starts its indices at 0, so its offset is shifted by r0 * cols / 8
    step = 16 if two_d else 1
    want_c, want_s, want_g = [], [], None
    for i in range(0, len(rows_out), step):
        r0 = rows_out[i]
        c, sc, g = o.quantize(w[r0:r0 + step], fmt, **{**kw, "given_amax": given,
                                                       "sr_offset": kw.get("sr_offset", 0) + (r0 * w.shape[1]) // 8})
        want_c.extend(c)
        want_s.extend(sc)
        want_g = g
    return np.array(want_c), np.array(want_s), want_g, rows_out


def _check_quant_rows(x_np, q: fp4.QTensor, params_oracle, rows_out, label):
    """Sampled output rows of q bit for bit against the oracle; returns the
    oracle's (codes, scales, g, rows)."""
    want_c, want_s, want_g, rows_out = _oracle_rows(x_np, q.fmt, params_oracle, rows_out)
    codes = q.codes.cpu().numpy()
    nsf = q.k // fp4.BLOCK[q.fmt]
    scales = untile_scales(q.scales.cpu().numpy(), q.rows, nsf)
    assert np.array_equal(scales[rows_out], want_s), mismatch_report(scales[rows_out], want_s, label + " scales")
    assert np.array_equal(codes[rows_out], want_c), mismatch_report(codes[rows_out], want_c, label + " codes")
    if want_g is not None:
        got_g = q.tensor_scale.cpu().numpy()[0]
        assert np.float32(got_g).view(np.uint32) == np.float32(want_g).view(np.uint32)
    return want_c, want_s, want_g, rows_out


def _check_gemm_sampled(a, b, y, fmt, out_bf16, label):
    """y[rows_a][:, rows_b] against the oracle's GEMM of the oracle's own
    quantizations of those rows of A and B (each a tuple from _check_quant_rows,
    which has already compared them with the GPU's codes).  Nothing of the GPU's
    output enters the expected values."""
    ca, sa, ga, ra = a
    cb, sb, gb, rb = b
    yr, bound = o.gemm(ca, sa, cb, sb, OF[fmt], ga, gb)
    got = y[torch.from_numpy(ra).to(y.device)][:, torch.from_numpy(rb).to(y.device)].float().cpu().numpy()
    got = got.astype(np.float64)
    tol = o.gemm_tolerance(bound, yr, out_bf16)
    bad = np.abs(got - yr) > tol
    assert not bad.any(), f"{label}: {bad.sum()} of {bad.size} sampled outputs outside the bound"


def test_linear_fprop_small_full():
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.linear_fprop_small()
    x, w = d["X"], d["W"]
    qx = fp4.fp4_quantize(x.cuda(), fp4.quant_params(MX))
    qw = fp4.fp4_quantize(w.cuda(), fp4.quant_params(MX))
    y = fp4.fp4_gemm(qx, qw, torch.float32)
    cx, sx, _ = o.quantize(x.float().numpy(), o.MXFP4)
    cw, sw, _ = o.quantize(w.float().numpy(), o.MXFP4)
    assert np.array_equal(qx.codes.cpu().numpy(), cx) and np.array_equal(qw.codes.cpu().numpy(), cw)
    yr, bound = o.gemm(cx, sx, cw, sw, o.MXFP4)
    assert np.all(np.abs(y.cpu().numpy() - yr) <= 1e-3 * bound)


def test_nvfp4_square_quantize_sr_dge():
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.nvfp4_square()
    t, dy = d["T"], d["dy"]
    tn = t.float().numpy()
    rows = _sample_rows(4096, 24, 1)
    for rnd, name in ((fp4.FP4_ROUND_RTN, "rtn"), (fp4.FP4_ROUND_SR, "sr")):
        q = fp4.fp4_quantize(t.cuda(), fp4.quant_params(NV, rnd, sr_seed=1))
        _check_quant_rows(tn, q, {"rounding": name, "sr_seed": 1}, rows, f"nvfp4 4096^2 {name}")
    # dequantize and DGE on the sampled rows
    q = fp4.fp4_quantize(t.cuda(), fp4.quant_params(NV))
    deq = fp4.fp4_dequantize(q, torch.float32).cpu().numpy()
    dx = fp4.fp4_dge_backward(t.cuda(), q, dy.cuda(), 5.0, 3.0).cpu().numpy()
    g = q.tensor_scale.cpu().numpy()[0]
    sc = untile_scales(q.scales.cpu().numpy(), 4096, 256)
    codes = q.codes.cpu().numpy()
    want = o.dequantize(codes[rows], sc[rows], o.NVFP4, g)
    assert np.array_equal(deq[rows].view(np.uint32), want.view(np.uint32))
    wdx = o.dge_backward(tn[rows], sc[rows], o.NVFP4, g, dy.float().numpy()[rows], 5.0, 3.0)
    assert np.all(np.abs(dx[rows] - wdx) <= 1e-6 * np.abs(wdx))


def test_llama1b_mlp_up_step():
    """The benchmark's step, op for op, checked on sampled rows."""
    import bench
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.llama1b_mlp_up()
    X, W, dY = (d[k].cuda() for k in ("X", "W", "dY"))
    step = bench.Step(fp4, X, W, dY, torch.device("cuda"))
    step.run(0, side=torch.cuda.Stream())        # the two-stream schedule the bench times
    torch.cuda.synchronize()
    assert fp4.fp4_sync_status() == 0 and fp4.fp4_sync_status(step.side_ctx) == 0
    xn, wn, dyn = (d[k].float().numpy() for k in ("X", "W", "dY"))
    off = 0                                      # step 0: sr_offset = 0
    r_m = _sample_rows(bench.M, 6, 2)
    r_n = _sample_rows(bench.N, 6, 3)
    r_k = _sample_rows(bench.K, 6, 4)
    # rows of each B operand, i.e. the sampled output columns of its GEMM
    r_nb = _sample_rows(bench.N, 24, 13)
    r_kb = _sample_rows(bench.K, 24, 14)
    sr = {"rounding": "sr", "rht": True, "sr_seed": 2, "rht_seed": 2, "sr_offset": off}
    xa = _check_quant_rows(xn, step.xq, {}, r_m, "fwd X")
    wb = _check_quant_rows(wn, step.wq, {}, r_nb, "fwd W")
    _check_quant_rows(wn, step.wq, {}, r_n, "fwd W rows")
    dya = _check_quant_rows(dyn, step.dyq_n, {**sr, "sr_stream": 0}, r_m, "dY rows")
    dyma = _check_quant_rows(dyn, step.dyq_m, {**sr, "sr_stream": 2, "transpose": True}, r_n, "dY cols")
    wtb = _check_quant_rows(wn, step.wq_t, {**sr, "sr_stream": 1, "transpose": True, "scaling": "2d"}, r_kb, "W 2d t")
    xtb = _check_quant_rows(xn, step.xq_t, {**sr, "sr_stream": 3, "transpose": True}, r_kb, "X t")
    _check_gemm_sampled(xa, wb, step.Y, NV, True, "fprop")
    _check_gemm_sampled(dya, wtb, step.dX, NV, True, "dgrad")
    _check_gemm_sampled(dyma, xtb, step.dW, NV, False, "wgrad")
    # DGE on the sampled rows of W
    sc = untile_scales(step.wq.scales.cpu().numpy(), bench.N, bench.K // 16)
    g = step.wq.tensor_scale.cpu().numpy()[0]
    dw = step.dW.cpu().numpy()
    want = o.dge_backward(wn[r_n], sc[r_n], o.NVFP4, g, dw[r_n], 5.0, 3.0)
    got = step.dWd.cpu().numpy()[r_n]
    assert np.all(np.abs(got - want) <= 1e-6 * np.abs(want))
    # the sigmoid-smoothed estimator in DGE's place, in the launch the bench times
    from test_gpu_soft import grad_tolerance, value_tolerance
    xs = o.scaled_inputs(wn[r_n], sc[r_n], o.NVFP4, g)
    for beta in (40.0, 1.0):
        got = fp4.fp4_soft_backward(step.W, step.wq, step.dW, beta).cpu().numpy()[r_n].astype(np.float64)
        want = o.soft_backward(wn[r_n], sc[r_n], o.NVFP4, g, dw[r_n], beta)
        assert np.all(np.abs(got - want) <= grad_tolerance(xs, beta, want, dw[r_n])), beta
    got = fp4.fp4_soft_forward(step.W, step.wq, 40.0).cpu().numpy()[r_n].astype(np.float64)
    want = o.soft_forward(wn[r_n], sc[r_n], o.NVFP4, g, 40.0)
    sv = o.block_scales_expanded(sc[r_n], o.NVFP4, g).astype(np.float64)
    assert np.all(np.abs(got - want) <= value_tolerance(sv, want))


@pytest.mark.parametrize("two_d", [False, True])
def test_dual_quantize_many_tiles_ragged(two_d):
    """The dual NVFP4 quantizer's persistent tile loop: 4144 x 4208 (65 x 33 =
    2145 tiles of 64 x 128 for 1216 CTAs, so most CTAs prefetch a second tile
    while quantizing the first; the last tile row holds 48 rows and the last
    tile column 112 columns).  Row layout RTN (or SR + RHT), transposed layout
    SR + RHT (with 16 x 16 blocks when two_d), as the step quantizes X and W;
    sampled rows of both layouts, including the ragged edges, bit for bit."""
    R, C = 4144, 4208
    rng = np.random.default_rng(71 + two_d)
    x = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-2, 2, (R, 1)))).astype(np.float32)
    x[:, rng.permutation(C)[:5]] *= 50
    xt = torch.from_numpy(x).to(torch.bfloat16)
    xn = xt.float().numpy()
    kr = dict(sr_seed=3, sr_stream=0, rht_seed=4, sr_offset=17 << 40)
    kc = dict(sr_seed=3, sr_stream=2, rht_seed=4, sr_offset=17 << 40)
    rows_sr = not two_d          # the W-like case keeps the row layout RTN
    pr = fp4.quant_params(NV, fp4.FP4_ROUND_SR if rows_sr else fp4.FP4_ROUND_RTN, rht=rows_sr, **kr)
    pc = fp4.quant_params(NV, fp4.FP4_ROUND_SR, fp4.FP4_SCALING_2D if two_d else fp4.FP4_SCALING_1D,
                          transpose=True, rht=True, **kc)
    qr, qc = fp4.fp4_quantize_dual(xt.cuda(), pr, pc)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([_sample_rows(R, 6, 5), [R - 48, R - 17, R - 2]]))
    cols = np.unique(np.concatenate([_sample_rows(C, 6, 6), [C - 112, C - 33, C - 2]]))
    if rows_sr:
        _check_quant_rows(xn, qr, {"rounding": "sr", "rht": True, **kr}, rows, "dual rows (SR + RHT)")
    else:
        _check_quant_rows(xn, qr, {}, rows, "dual rows (RTN)")
    pcol = {"rounding": "sr", "rht": True, "transpose": True, **kc}
    if two_d:
        pcol["scaling"] = "2d"
    _check_quant_rows(xn, qc, pcol, cols, "dual cols")


def test_ffn7b_step():
    """The 7B-shaped FFN step the benchmark times (MXFP4, RTN, bf16 out): X, W
    and dY each quantized in both layouts from one read, then fprop, dgrad and
    wgrad, in the benchmark's launch configuration.  Sampled rows of every
    quantized operand bit for bit; sampled rows x sampled columns of every GEMM
    against the oracle's GEMM of the oracle's quantization of the inputs."""
    import bench
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.ffn7b()
    X, W, dY = (d[k].cuda() for k in ("X", "W", "dY"))
    M, K = X.shape
    N = W.shape[0]
    step = bench.FfnStep(fp4, X, W, dY, torch.device("cuda"))
    step.run(0, side=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert fp4.fp4_sync_status() == 0 and fp4.fp4_sync_status(step.side_ctx) == 0
    xn, wn, dyn = (d[k].float().numpy() for k in ("X", "W", "dY"))
    r_m, r_n = _sample_rows(M, 4, 5), _sample_rows(N, 4, 6)
    r_nb, r_kb = _sample_rows(N, 24, 16), _sample_rows(K, 24, 17)
    t = {"transpose": True}
    xa = _check_quant_rows(xn, step.xq, {}, r_m, "7b X")
    wb = _check_quant_rows(wn, step.wq, {}, r_nb, "7b W")
    dya = _check_quant_rows(dyn, step.dyq_n, {}, r_m, "7b dY rows")
    wtb = _check_quant_rows(wn, step.wq_t, t, r_kb, "7b W t")
    dyma = _check_quant_rows(dyn, step.dyq_m, t, r_n, "7b dY cols")
    xtb = _check_quant_rows(xn, step.xq_t, t, r_kb, "7b X t")
    _check_gemm_sampled(xa, wb, step.Y, MX, True, "7b fprop")
    _check_gemm_sampled(dya, wtb, step.dX, MX, True, "7b dgrad")
    _check_gemm_sampled(dyma, xtb, step.dW, MX, True, "7b wgrad")


def _oracle_channel_errors(xn, chunk=1024):
    """e_c over all rows of xn (NVFP4, the full tensor's amax), by the oracle,
    one row chunk at a time (fp64 sums)."""
    amax = o.tensor_amax(xn)
    g = o.nvfp4_tensor_scale(amax)
    e = np.zeros(xn.shape[1], np.float64)
    for r0 in range(0, xn.shape[0], chunk):
        part = xn[r0:r0 + chunk]
        c, sc, _ = o.quantize(part, o.NVFP4, given_amax=amax)
        e += o.hcp_channel_errors(part, c, sc, o.NVFP4, g)
    return e


def test_hcp_square_full():
    """Hot-channel selection and the compensated GEMM (bf16 and MXFP8 extra columns)
    at the benchmark's size.
    The GPU's hot set equals the oracle's outside a 1e-5 relative band around
    the h-th largest error (inside it the fp32 sums may order channels
    differently); the GEMM then runs on the oracle's set and is compared on
    sampled rows x columns with the oracle's product of the oracle's
    quantizations."""
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.hcp_square()
    X, W = d["X"].cuda(), d["W"].cuda()
    M, K = X.shape
    h = fp4.fp4_hcp_num_hot(K)
    assert h == 369
    qx = fp4.fp4_quantize(X, fp4.quant_params(NV))
    qw = fp4.fp4_quantize(W, fp4.quant_params(NV))
    hot = fp4.fp4_hcp_select(X, qx, h).cpu().numpy()
    xfull = d["X"].float().numpy()
    e = _oracle_channel_errors(xfull)
    hot_o = o.hcp_top_channels(e, h)
    assert set(d["hot_cols"].tolist()) <= set(hot_o.tolist())
    t = np.sort(e)[::-1][h - 1]
    sure_in = set(np.nonzero(e > t * (1 + 1e-5))[0].tolist())
    sure_out = set(np.nonzero(e < t * (1 - 1e-5))[0].tolist())
    got = set(hot.tolist())
    assert sure_in <= got and not (got & sure_out)
    hot_t = torch.from_numpy(hot_o).cuda()
    y1 = fp4.fp4_hcp_gemm(X, W, qx, qw, hot_t, h, fp4.FP4_HCP_SINGLE, 2, torch.float32)
    y2 = fp4.fp4_hcp_gemm(X, W, qx, qw, hot_t, h, fp4.FP4_HCP_TWO, 2, torch.float32)
    y3 = fp4.fp4_hcp_gemm(X, W, qx, qw, hot_t, h, fp4.FP4_HCP_SINGLE_MXFP8, 2, torch.float32)
    wn = d["W"].float().numpy()
    cx, sx, gx, rows = _check_quant_rows(xfull, qx, {}, _sample_rows(M, 3, 7), "hcp X")
    cw, sw, gw, cols = _check_quant_rows(wn, qw, {}, _sample_rows(W.shape[0], 24, 8), "hcp W")
    yr, bound = o.hcp_gemm(xfull[rows], cx, sx, wn[cols], cw, sw, o.NVFP4, gx, gw, hot_o, 2)
    for y, label in ((y1, "single"), (y2, "two")):
        got_y = y.cpu().numpy()[rows][:, cols].astype(np.float64)
        assert np.all(np.abs(got_y - yr) <= 1e-3 * bound), label
    # the MXFP8 extra columns: the oracle's product with the same MXFP8 values
    y3r, bound3 = o.hcp_gemm_mxfp8(xfull[rows], cx, sx, wn[cols], cw, sw, o.NVFP4, gx, gw, hot_o, 2)
    got3 = y3.cpu().numpy()[rows][:, cols].astype(np.float64)
    assert np.all(np.abs(got3 - y3r) <= o.gemm_tolerance(bound3, y3r, False)), "single mxfp8"


def test_hcp_square_variants_full():
    """Hot channels zeroed (single kernel) and the E4M3 residual GEMM, at the bench's size."""
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.hcp_square()
    X, W = d["X"].cuda(), d["W"].cuda()
    M, K = X.shape
    h = fp4.fp4_hcp_num_hot(K)
    qx = fp4.fp4_quantize(X, fp4.quant_params(NV))
    qw = fp4.fp4_quantize(W, fp4.quant_params(NV))
    hot = fp4.fp4_hcp_select(X, qx, h)
    hot_np = hot.cpu().numpy()
    x0q = fp4.fp4_hcp_quantize_zeroed(X, fp4.quant_params(NV), hot, h)
    y0 = fp4.fp4_hcp_gemm(X, W, x0q, qw, hot, h, fp4.FP4_HCP_SINGLE, 0, torch.bfloat16)
    y8 = fp4.fp4_hcp_gemm(X, W, qx, qw, hot, h, fp4.FP4_HCP_TWO_FP8, 2, torch.bfloat16)
    xfull = d["X"].float().numpy()
    # the zeroed tensor's scale from the whole tensor
    x0 = o.hcp_zero_columns(xfull, hot_np)
    g0 = o.nvfp4_tensor_scale(o.tensor_amax(x0))
    assert np.float32(x0q.tensor_scale.cpu().numpy()[0]).view(np.uint32) == np.float32(g0).view(np.uint32)
    rows = _sample_rows(M, 3, 8)
    wn = d["W"].float().numpy()
    cw = qw.codes.cpu().numpy()
    sw = untile_scales(qw.scales.cpu().numpy(), W.shape[0], K // 16)
    gw = qw.tensor_scale.cpu().numpy()[0]
    # zeroed: codes of the sampled rows bit-exact, then the GEMM bound
    wc, ws, _ = o.quantize(x0[rows], o.NVFP4, given_amax=o.tensor_amax(x0))
    c0 = x0q.codes.cpu().numpy()[rows]
    s0 = untile_scales(x0q.scales.cpu().numpy(), M, K // 16)[rows]
    assert np.array_equal(c0, wc) and np.array_equal(s0, ws)
    y, bound = o.gemm(c0, s0, cw, sw, o.NVFP4, g0, gw)
    a_ext, b_ext = o.hcp_zeroed_operands(xfull[rows], wn, o.NVFP4, g0, gw, hot_np)
    alpha32 = float(np.float32(np.float32(g0) * np.float32(gw)))
    y = y + alpha32 * (a_ext.astype(np.float64) @ b_ext.astype(np.float64).T)
    bound = bound + alpha32 * (np.abs(a_ext.astype(np.float64)) @ np.abs(b_ext.astype(np.float64)).T)
    got = y0.float().cpu().numpy()[rows].astype(np.float64)
    assert np.all(np.abs(got - y) <= o.gemm_tolerance(bound, y, True)), "zeroed"
    # E4M3 residual (two kernels, order 2)
    cx = qx.codes.cpu().numpy()[rows]
    sx = untile_scales(qx.scales.cpu().numpy(), M, K // 16)[rows]
    gx = qx.tensor_scale.cpu().numpy()[0]
    yr, bound = o.hcp_gemm_fp8(xfull[rows], cx, sx, wn, cw, sw, o.NVFP4, gx, gw, hot_np, 2)
    got = y8.float().cpu().numpy()[rows].astype(np.float64)
    tol = o.gemm_tolerance(bound, yr, True) + 2.0 ** -8 * np.abs(yr)
    assert np.all(np.abs(got - yr) <= tol), "fp8"


def test_occ_full():
    """Outlier clamping and compensation at the bench's size (X 16384x4096, W 4096^2, NVFP4)."""
    import bench
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.hcp_square(bench.OCC_M, bench.OCC_K, bench.OCC_N)
    X, W = d["X"].cuda(), d["W"].cuda()
    M, K = X.shape
    tau, n_out = fp4.fp4_occ_threshold(X)
    counts = torch.empty((K,), dtype=torch.float32, device="cuda")
    xq = fp4.fp4_occ_quantize(X, fp4.quant_params(NV), tau, col_counts=counts)
    wq = fp4.fp4_quantize(W, fp4.quant_params(NV))
    y = fp4.fp4_occ_gemm(X, W, xq, wq, tau, counts, bench.OCC_DENSE, fp4.fp4_occ_max_outliers(M, K))
    assert fp4.fp4_sync_status() == 0
    xfull = d["X"].float().numpy()
    a = np.abs(xfull).reshape(-1)
    rank = int(np.ceil(0.99 * a.size))
    t = np.float32(np.partition(a, rank - 1)[rank - 1])       # the nearest-rank order statistic
    assert tau.item() == float(t)
    out = np.abs(xfull) > t
    assert n_out.item() == int(out.sum())
    assert np.array_equal(counts.cpu().numpy(), out.sum(axis=0).astype(np.float32))
    rows = _sample_rows(M, 3, 9)
    xc, dx = o.occ_split(xfull[rows], t)
    wc, ws, _ = o.quantize(xc, o.NVFP4, given_amax=t)
    c = xq.codes.cpu().numpy()[rows]
    s = untile_scales(xq.scales.cpu().numpy(), M, K // 16)[rows]
    assert np.array_equal(c, wc) and np.array_equal(s, ws)
    g = xq.tensor_scale.cpu().numpy()[0]
    wn = d["W"].float().numpy()
    cw = wq.codes.cpu().numpy()
    sw = untile_scales(wq.scales.cpu().numpy(), W.shape[0], K // 16)
    gw = wq.tensor_scale.cpu().numpy()[0]
    yr, bound = o.gemm(c, s, cw, sw, o.NVFP4, g, gw)
    dxf = dx.astype(np.float64)
    comp = np.abs(dxf) @ np.abs(wn.astype(np.float64)).T
    yr = yr + dxf @ wn.astype(np.float64).T
    tol = 1e-3 * (bound + comp) + 2.0 ** -8 * comp + 2.0 ** -8 * (np.abs(yr) + comp)
    got = y.float().cpu().numpy()[rows].astype(np.float64)
    assert np.all(np.abs(got - yr) <= tol)


@pytest.mark.parametrize("fmt", [NV, MX])
def test_block_sizes_full(fmt):
    """Blocks of 16-128 on the step's X (8192 x 2048), sampled rows bit-exact."""
    from fp4_block_scaled_e8m0_gb300 import inputs
    x = inputs.llama1b_mlp_up()["X"]
    xn = x.float().numpy()
    rows = _sample_rows(x.shape[0], 4, 10)
    g = o.nvfp4_tensor_scale(o.tensor_amax(xn)) if fmt == NV else None
    for block in (16, 32, 64, 128):
        p = fp4.quant_params(fmt, sf_layout=fp4.FP4_SF_ROWMAJOR, block=block)
        q = fp4.fp4_quantize(x.cuda(), p)
        wc, ws, _ = o.quantize(xn[rows], OF[fmt], block=block, given_amax=o.tensor_amax(xn))
        nsf = x.shape[1] // block
        sc = q.scales.cpu().numpy()[: x.shape[0] * nsf].reshape(x.shape[0], nsf)[rows]
        assert np.array_equal(sc, ws), block
        assert np.array_equal(q.codes.cpu().numpy()[rows], wc), block
        if g is not None:
            assert np.float32(q.tensor_scale.cpu().numpy()[0]).view(np.uint32) == np.float32(g).view(np.uint32)
