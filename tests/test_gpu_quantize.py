"""GPU <-> oracle parity for the quantization-side kernels, through the C ABI.

Codes, scales, tensor scales, RHT outputs and stochastic-rounding codes must
match the oracle bit for bit; the DGE backward within 1e-6 relative.
Sizes span several tiles and end in ragged tails.
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o
from _util import mismatch_report, np32, untile_scales

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


def _input(shape, seed, dtype=torch.bfloat16, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    x *= np.exp(rng.uniform(-3, 3, (shape[0], 1))).astype(np.float32)     # rows of very different scale
    if outliers:
        cols = rng.permutation(shape[1])[:3]
        x[:, cols] *= 100
    x[0, :5] = 0.0
    x[1, :16] = 0.0                                                          # an all-zero block
    x[2, 3] = -0.0
    t = torch.from_numpy(x).to(dtype)
    return t, t.float().numpy()


def _gpu_quant_np(q: fp4.QTensor):
    codes = q.codes.cpu().numpy()
    nsf = q.k // fp4.BLOCK[q.fmt]
    sc = q.scales.cpu().numpy()
    scales = untile_scales(sc, q.rows, nsf) if q.sf_layout == fp4.FP4_SF_MMA else sc[: q.rows * nsf].reshape(q.rows, nsf)
    g = q.tensor_scale.cpu().numpy()[0] if q.tensor_scale is not None else None
    return codes, scales, g


def _check_quant(q, want, label):
    codes, scales, g = _gpu_quant_np(q)
    wc, ws, wg = want
    assert np.array_equal(scales, ws), mismatch_report(scales, ws, label + " scales")
    assert np.array_equal(codes, wc), mismatch_report(codes, wc, label + " codes")
    if wg is not None:
        assert np.float32(g).view(np.uint32) == np.float32(wg).view(np.uint32), (label, g, wg)


# ---------------------------------------------------------------------------
# element encoders
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("method", [0, 1])
def test_encode_e2m1_matches_oracle(method):
    bits = np.arange(65536, dtype=np.uint32) << 16
    base = bits.view(np.float32)
    base = base[np.isfinite(base)]
    xs = np.concatenate([(base * np.float32(m)).astype(np.float32) for m in (1.0, 4.0, 0.03125, 1.0 / 3.0)])
    xs = xs[np.isfinite(xs)]
    got = fp4.fp4_encode_e2m1(torch.from_numpy(xs).cuda(), method).cpu().numpy()
    want = o.e2m1_encode_rtn(xs)
    assert np.array_equal(got, want), mismatch_report(got, want, f"e2m1 method {method}")


def test_encode_e4m3_matches_oracle():
    table = o.E4M3_VALUES[:127]
    mids = (table[1:] + table[:-1]) / 2
    rng = np.random.default_rng(1)
    t = np.concatenate([table, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), rng.uniform(0, 500, 100000),
                        np.exp(rng.uniform(-14, 7, 100000)), [449.0, 464.0, 1e9]]).astype(np.float32)
    got = fp4.fp4_encode_e4m3(torch.from_numpy(t).cuda()).cpu().numpy()
    want = o.e4m3_encode_rn_satfinite(t)
    assert np.array_equal(got, want), mismatch_report(got, want, "e4m3")


# ---------------------------------------------------------------------------
# quantize: rows (blocks along cols)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("rounding", [fp4.FP4_ROUND_RTN, fp4.FP4_ROUND_SR])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
def test_quantize_rows(fmt, rounding, rht, dtype, sf_layout):
    x, xn = _input((200, 320), seed=10 + fmt, dtype=dtype)
    x = x.cuda()
    kw = dict(sr_seed=0x1234_5678_9, sr_offset=17, sr_stream=5, rht_seed=2)
    q = fp4.fp4_quantize(x, fp4.quant_params(fmt, rounding, rht=rht, sf_layout=sf_layout, **kw))
    want = o.quantize(xn, FMT[fmt], "sr" if rounding else "rtn", rht=rht, **kw)
    _check_quant(q, want, f"rows fmt={fmt} sr={rounding} rht={rht}")


def test_quantize_given_amax_and_zero_tensor():
    x, xn = _input((64, 128), seed=3)
    x = x.cuda()
    amax = torch.tensor([1000.0], device="cuda")
    q = fp4.fp4_quantize(x, fp4.quant_params(fp4.FP4_FMT_NVFP4), given_amax=amax)
    _check_quant(q, o.quantize(xn, o.NVFP4, given_amax=1000.0), "given amax")
    z = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    qz = fp4.fp4_quantize(z, fp4.quant_params(fp4.FP4_FMT_NVFP4))
    _check_quant(qz, o.quantize(np.zeros((32, 64), np.float32), o.NVFP4), "zero tensor")


# ---------------------------------------------------------------------------
# quantize: transposed (blocks along rows), 2D, dual
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("rounding", [fp4.FP4_ROUND_RTN, fp4.FP4_ROUND_SR])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_transposed(fmt, rounding, rht, dtype):
    x, xn = _input((320, 200), seed=20 + fmt, dtype=dtype)
    x = x.cuda()
    kw = dict(sr_seed=77, sr_offset=3, sr_stream=2, rht_seed=9)
    q = fp4.fp4_quantize(x, fp4.quant_params(fmt, rounding, transpose=True, rht=rht, **kw))
    want = o.quantize(xn, FMT[fmt], "sr" if rounding else "rtn", transpose=True, rht=rht, **kw)
    _check_quant(q, want, f"cols fmt={fmt} sr={rounding} rht={rht}")


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("rounding", [fp4.FP4_ROUND_RTN, fp4.FP4_ROUND_SR])
@pytest.mark.parametrize("rht", [False, True])
def test_quantize_2d(transpose, rounding, rht):
    x, xn = _input((320, 208), seed=30)
    x = x.cuda()
    kw = dict(sr_seed=2, sr_offset=0, sr_stream=1, rht_seed=2)
    q = fp4.fp4_quantize(x, fp4.quant_params(fp4.FP4_FMT_NVFP4, rounding, fp4.FP4_SCALING_2D, transpose, rht, **kw))
    want = o.quantize(xn, o.NVFP4, "sr" if rounding else "rtn", "2d", transpose, rht, **kw)
    _check_quant(q, want, f"2d t={transpose} sr={rounding} rht={rht}")


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("rounding", [fp4.FP4_ROUND_RTN, fp4.FP4_ROUND_SR])
@pytest.mark.parametrize("rht", [False, True])
def test_quantize_dual(fmt, rounding, rht):
    x, xn = _input((320, 224), seed=40 + fmt)
    x = x.cuda()
    pr = fp4.quant_params(fmt, rounding, rht=rht, sr_seed=2, sr_stream=0, rht_seed=2)
    pc = fp4.quant_params(fmt, rounding, transpose=True, rht=rht, sr_seed=2, sr_stream=2, rht_seed=2)
    qr, qc = fp4.fp4_quantize_dual(x, pr, pc)
    mode = "sr" if rounding else "rtn"
    _check_quant(qr, o.quantize(xn, FMT[fmt], mode, rht=rht, sr_seed=2, sr_stream=0, rht_seed=2), "dual rows")
    _check_quant(qc, o.quantize(xn, FMT[fmt], mode, transpose=True, rht=rht, sr_seed=2, sr_stream=2, rht_seed=2),
                 "dual cols")


# Mixed parameters per layout, as a training step uses them: X and W go to the
# forward GEMM with RTN and to a backward GEMM with SR + RHT (W also with 16x16
# 2D blocks); each output must equal its own single-layout quantization.
@pytest.mark.parametrize("case", ["x_fwd_bwd", "w_fwd_bwd2d", "rows2d_cols1d"])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
def test_quantize_dual_mixed(case, sf_layout):
    x, xn = _input((336, 208), seed=44)
    x = x.cuda()
    NV, RTN, SR, D1, D2 = fp4.FP4_FMT_NVFP4, fp4.FP4_ROUND_RTN, fp4.FP4_ROUND_SR, fp4.FP4_SCALING_1D, fp4.FP4_SCALING_2D
    row_cfg, col_cfg = {
        "x_fwd_bwd": ((RTN, D1, False), (SR, D1, True)),
        "w_fwd_bwd2d": ((RTN, D1, False), (SR, D2, True)),
        "rows2d_cols1d": ((RTN, D2, False), (RTN, D1, False)),
    }[case]
    kr = dict(sr_seed=7, sr_offset=3, sr_stream=1, rht_seed=5)
    kc = dict(sr_seed=7, sr_offset=3, sr_stream=2, rht_seed=5)
    pr = fp4.quant_params(NV, row_cfg[0], row_cfg[1], rht=row_cfg[2], sf_layout=sf_layout, **kr)
    pc = fp4.quant_params(NV, col_cfg[0], col_cfg[1], transpose=True, rht=col_cfg[2], sf_layout=sf_layout, **kc)
    qr, qc = fp4.fp4_quantize_dual(x, pr, pc)
    mode = {RTN: "rtn", SR: "sr"}
    sc = {D1: "1d", D2: "2d"}
    _check_quant(qr, o.quantize(xn, o.NVFP4, mode[row_cfg[0]], sc[row_cfg[1]], False, row_cfg[2], **kr), case + " rows")
    _check_quant(qc, o.quantize(xn, o.NVFP4, mode[col_cfg[0]], sc[col_cfg[1]], True, col_cfg[2], **kc), case + " cols")


# ---------------------------------------------------------------------------
# tiny and subnormal blocks
# ---------------------------------------------------------------------------
def _tiny_input(shape, seed, fmt):
    """bf16 values far below 1.  MXFP4: rows scaled by 2^u, u in [-150, -100],
    so that whole rows and blocks are bf16 subnormals (below 2^-126) or flush
    to zero in bf16, and others straddle the smallest normal; row 0 holds the
    hand-derived blocks of tests/golden/mxfp4_tiny_blocks.txt.  NVFP4: rows
    scaled by 2^u, u in [-140, -100], with one element 2^-100, the tensor amax:
    the tensor scale stays normal, blocks near 2^-110 keep small E4M3 scales and
    the subnormal blocks get scale 0 (all codes 0)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float64)
    lo = -150 if fmt == fp4.FP4_FMT_MXFP4 else -140
    x *= np.exp2(rng.uniform(lo, -100, (shape[0], 1)))
    if fmt == fp4.FP4_FMT_MXFP4:
        from conftest import golden
        rows = golden("mxfp4_tiny_blocks.txt")
        blocks = sorted({r[0] for r in rows})
        x[0, : 32 * len(blocks)] = 0.0
        for r in rows:
            if r[1] != "scale":
                x[0, 32 * blocks.index(r[0]) + int(r[1])] = float.fromhex(r[2])
    else:
        x = np.clip(x, -2.0 ** -101, 2.0 ** -101)
        x[3, 17] = 2.0 ** -100
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t, t.float().numpy()


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("rounding", [fp4.FP4_ROUND_RTN, fp4.FP4_ROUND_SR])
@pytest.mark.parametrize("layout", ["rows", "cols", "dual"])
def test_quantize_tiny_blocks(fmt, rounding, layout):
    """Codes and scales of tiny / bf16-subnormal blocks, bit for bit: the E8M0
    clamp, the subnormal amax's true exponent, no flush to zero of subnormal
    inputs or of the 2^-127 scale; then the dequantized values (fp32 and bf16)."""
    x, xn = _tiny_input((160, 288), 90 + fmt, fmt)
    assert np.count_nonzero(np.abs(xn) < 2.0 ** -126) > 1000            # subnormals are present
    x = x.cuda()
    mode = "sr" if rounding else "rtn"
    kw = dict(sr_seed=11, sr_offset=5, sr_stream=3)
    pr = fp4.quant_params(fmt, rounding, **kw)
    pc = fp4.quant_params(fmt, rounding, transpose=True, **kw)
    outs = []
    if layout == "rows":
        outs.append((fp4.fp4_quantize(x, pr), False))
    elif layout == "cols":
        outs.append((fp4.fp4_quantize(x, pc), True))
    else:
        qr, qc = fp4.fp4_quantize_dual(x, pr, pc)
        outs += [(qr, False), (qc, True)]
    for q, tr in outs:
        want = o.quantize(xn, FMT[fmt], mode, transpose=tr, **kw)
        _check_quant(q, want, f"tiny {layout} t={tr} fmt={fmt} {mode}")
        for out_dtype in (torch.float32, torch.bfloat16):
            got = fp4.fp4_dequantize(q, out_dtype).float().cpu().numpy()
            wd = o.dequantize(want[0], want[1], FMT[fmt], want[2])
            if out_dtype == torch.bfloat16:
                wd = o.bf16_round(wd)
            assert np.array_equal(got.view(np.uint32), wd.view(np.uint32)), \
                mismatch_report(got.view(np.uint32), wd.view(np.uint32), f"tiny dequant {out_dtype}")
        if fmt == fp4.FP4_FMT_MXFP4 and not tr:
            # the hand-derived blocks: row 0, blocks 0..2 (bytes 0, 0, 1)
            _, sc, _ = _gpu_quant_np(q)
            assert sc[0, :3].tolist() == [0, 0, 1]


@pytest.mark.parametrize("axis", [-1, 0, 1])
@pytest.mark.parametrize("shape", [(320, 208), (48, 40)])
def test_amax(axis, shape):
    if axis == 1 and shape[1] % 16:
        pytest.skip("row transform needs cols % 16")
    x, xn = _input(shape, seed=50, outliers=False)
    got = fp4.fp4_amax(x.cuda(), axis, 3).cpu().numpy()[0]
    w = xn if axis < 0 else o.rht16(xn, axis, 3)
    assert np.float32(got) == o.tensor_amax(w)


# ---------------------------------------------------------------------------
# dequantize, RHT, DGE
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
def test_dequantize(fmt, out_dtype, sf_layout):
    x, xn = _input((200, 320), seed=60)
    q = fp4.fp4_quantize(x.cuda(), fp4.quant_params(fmt, sf_layout=sf_layout))
    got = fp4.fp4_dequantize(q, out_dtype).float().cpu().numpy()
    c, s, g = o.quantize(xn, FMT[fmt])
    want = o.dequantize(c, s, FMT[fmt], g)
    if out_dtype == torch.bfloat16:
        want = o.bf16_round(want)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), mismatch_report(got, want, "dequant")


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rht16_bit_exact(axis, dtype):
    x, xn = _input((96, 208), seed=70, dtype=dtype)
    got = fp4.fp4_rht16(x.cuda(), axis, 2).cpu().numpy()
    want = o.rht16(xn, axis, 2)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), mismatch_report(got, want, "rht16")


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
@pytest.mark.parametrize("outside", [1.0, 0.0])
def test_dge_backward(fmt, sf_layout, outside):
    x, xn = _input((200, 320), seed=80)
    rng = np.random.default_rng(81)
    dy = torch.from_numpy(rng.standard_normal((200, 320)).astype(np.float32)).to(torch.bfloat16)
    q = fp4.fp4_quantize(x.cuda(), fp4.quant_params(fmt, sf_layout=sf_layout))
    got = fp4.fp4_dge_backward(x.cuda(), q, dy.cuda(), k=5.0, clamp=3.0, outside=outside).cpu().numpy()
    _, s, g = o.quantize(xn, FMT[fmt])
    want = o.dge_backward(xn, s, FMT[fmt], g, dy.float().numpy(), 5.0, 3.0, outside)
    err = np.abs(got.astype(np.float64) - want)
    bad = err > 1e-6 * np.abs(want)
    assert not bad.any(), f"{bad.sum()} elements off; worst rel {np.max(err / np.maximum(np.abs(want), 1e-30))}"
