"""GPU <-> oracle parity for block sizes 16-128 with either scale format
("深度学习中的梯度计算基础" §4.2) and the quality sums behind §5.1's relative-error
table, through the C ABI.

Codes, scales and the tensor scale bit-exact at every block size; the
dequantized values bit-exact; the fp64 quality sums of the dequantized
reconstruction within 1e-9 relative (summation order).  For the
sigmoid-smoothed reconstruction each value may differ from the oracle's by
delta = 1.5e-5 s + 2^-22 |x_hat| (the bound of the soft forward), so the sums may
move by sum(2 |e| delta + delta^2), sum(2 |x_hat| delta + delta^2) and
sum(|x| delta); the test takes those bounds from the oracle's own values.
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o
from _util import mismatch_report

pytestmark = pytest.mark.gpu

FMT = {fp4.FP4_FMT_MXFP4: o.MXFP4, fp4.FP4_FMT_NVFP4: o.NVFP4}
BLOCKS = [16, 32, 64, 128]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    from fp4_block_scaled_e8m0_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    fp4.load_library()


def _input(shape, seed, dtype=torch.bfloat16):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    x *= np.exp(rng.uniform(-3, 3, (shape[0], 1))).astype(np.float32)
    x[:, rng.permutation(shape[1])[:3]] *= 100
    x[1, :128] = 0.0
    t = torch.from_numpy(x).to(dtype)
    return t, t.float().numpy()


def _params(fmt, block, rounding="rtn", rht=False):
    rnd = fp4.FP4_ROUND_SR if rounding == "sr" else fp4.FP4_ROUND_RTN
    return fp4.quant_params(fmt, rnd, rht=rht, sf_layout=fp4.FP4_SF_ROWMAJOR, block=block, sr_seed=5, sr_stream=2,
                            sr_offset=9, rht_seed=4)


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("rounding,rht", [("rtn", False), ("sr", False), ("sr", True)])
def test_quantize_any_block(fmt, block, rounding, rht):
    x, xn = _input((333, 384), seed=70 + block)
    q = fp4.fp4_quantize(x.cuda(), _params(fmt, block, rounding, rht))
    wc, ws, wg = o.quantize(xn, FMT[fmt], rounding, rht=rht, sr_seed=5, sr_stream=2, sr_offset=9, rht_seed=4,
                            block=block)
    codes = q.codes.cpu().numpy()
    scales = q.scales.cpu().numpy()[: 333 * (384 // block)].reshape(333, 384 // block)
    assert np.array_equal(scales, ws), mismatch_report(scales, ws, "scales")
    assert np.array_equal(codes, wc), mismatch_report(codes, wc, "codes")
    if wg is not None:
        assert np.float32(q.tensor_scale.cpu().numpy()[0]).view(np.uint32) == np.float32(wg).view(np.uint32)
    deq = fp4.fp4_dequantize(q, out_dtype=torch.float32).cpu().numpy()
    want = o.dequantize(wc, ws, FMT[fmt], wg, block=block)
    assert np.array_equal(deq, want), mismatch_report(deq, want, "dequantized")


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("block", BLOCKS)
def test_quality_sums_any_block(fmt, block):
    x, xn = _input((200, 256), seed=80 + block)
    xd = x.cuda()
    q = fp4.fp4_quantize(xd, _params(fmt, block))
    c, s, g = o.quantize(xn, FMT[fmt], block=block)
    a = xn.astype(np.float64).reshape(-1)
    # dequantized reconstruction
    got, st = (t.cpu().numpy() for t in fp4.fp4_quant_error_stats(xd, q))
    h = o.dequantize(c, s, FMT[fmt], g, block=block).astype(np.float64).reshape(-1)
    want = np.array([a @ a, h @ h, a @ h, ((a - h) ** 2).sum()])
    assert np.allclose(got, want, rtol=1e-9, atol=0)
    rel = o.relative_error(xn, h)
    assert abs(fp4.stats_dict(st)["rel_err"] - rel) <= 1e-9 * rel
    # sigmoid-smoothed reconstruction
    for beta in (10.0, 40.0):
        got = fp4.fp4_quant_error_stats(xd, q, beta=beta)[0].cpu().numpy()
        hs = o.soft_forward(xn, s, FMT[fmt], g, beta, block=block).reshape(-1)
        sv = o.block_scales_expanded(s, FMT[fmt], g, block=block).astype(np.float64).reshape(-1)
        d = 1.5e-5 * sv + 2.0 ** -22 * np.abs(hs)
        e = a - hs
        want = np.array([a @ a, hs @ hs, a @ hs, e @ e])
        bound = np.array([1e-9 * (a @ a), (2 * np.abs(hs) * d + d * d).sum(), (np.abs(a) * d).sum(),
                          (2 * np.abs(e) * d + d * d).sum()]) + 1e-9 * np.abs(want)
        assert np.all(np.abs(got - want) <= bound), (beta, got, want, bound)


def test_other_blocks_are_quantize_only():
    x, _ = _input((128, 256), seed=90)
    q = fp4.fp4_quantize(x.cuda(), _params(fp4.FP4_FMT_NVFP4, 64))
    with pytest.raises(fp4.FP4Error):
        fp4.fp4_gemm(q, q)
    with pytest.raises(fp4.FP4Error):
        fp4.fp4_dge_backward(x.cuda(), q, x.cuda())
    with pytest.raises(fp4.FP4Error):                     # 64-blocks need row-major scales
        fp4.fp4_quantize(x.cuda(), fp4.quant_params(fp4.FP4_FMT_NVFP4, block=64))
