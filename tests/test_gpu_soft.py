"""GPU <-> oracle parity for the sigmoid-smoothed quantizer Q_soft ("深度学习中的梯度计算基础"
§3.2), forward value and backward estimator, through the C ABI.

Tolerances follow from the kernels' fp32 arithmetic (x / s itself is formed
bit-identically on both sides):

* each term's exponent beta |x/s - c| carries <= 4 roundings of 2^-24, so
  t = e^-z is off by <= 4 * 2^-24 * z relative, plus <= 2^-22 from ex2.approx;
* Q_soft': every term is a weighted share of the sum and the N / D fraction adds
  <= (4 * 14 + 3) roundings, so the relative error is below
  1e-5 + 5e-7 (z_near + 3), z_near = beta * distance to the nearest threshold
  (twice the estimate above; the + 3 covers the spread of the weights when beta
  is small), plus the window's left-out terms (< 2^-23), plus terms below
  fp32's normal range flushed to 0 (< beta * 12 * 2^-126 absolute);
* Q_soft: each of <= 14 terms adds <= 7.2e-7 (sigma's exponent error, the
  approximate division, the running sum's rounding), so |error| <= 1.5e-5 in
  units of the block scale, plus the final rounding of y.
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o

pytestmark = pytest.mark.gpu

FMT = {fp4.FP4_FMT_MXFP4: o.MXFP4, fp4.FP4_FMT_NVFP4: o.NVFP4}
# one beta in each evaluation window (all thresholds; 4, 2, 1 per side) and the
# window boundaries
BETAS = [0.5, 5.0, 9.71, 12.0, 19.41, 25.0, 38.82, 40.0, 100.0]


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
    cols = rng.permutation(shape[1])[:3]
    x[:, cols] *= 100                                        # outlier columns
    x[1, :32] = 0.0                                          # all-zero blocks
    x[2, 3] = -0.0
    t = torch.from_numpy(x).to(dtype)
    return t, t.float().numpy()


def _dist_to_threshold(xs):
    c = o.soft_grid()[1]
    return np.abs(np.abs(np.asarray(xs, np.float64))[..., None] - c[7:]).min(axis=-1)


def grad_tolerance(xs, beta, want, dy):
    z_near = beta * _dist_to_threshold(xs)
    rel = 1e-5 + 5e-7 * (z_near + 3.0) + 2.0 ** -23
    return np.abs(dy) * (rel * np.abs(want / np.where(dy == 0, 1, dy)) + beta * 12 * 2.0 ** -126) \
        + 2.0 ** -24 * np.abs(want)


def value_tolerance(s, want):
    return 1.5e-5 * s + 2.0 ** -22 * np.abs(want)


def _quantized(x, fmt, sf_layout):
    q = fp4.fp4_quantize(x.cuda(), fp4.quant_params(fmt, sf_layout=sf_layout))
    return q


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
@pytest.mark.parametrize("beta", BETAS)
def test_soft_backward(fmt, sf_layout, beta):
    x, xn = _input((333, 320), seed=90)
    rng = np.random.default_rng(91)
    dy = torch.from_numpy(rng.standard_normal((333, 320)).astype(np.float32)).to(torch.bfloat16)
    q = _quantized(x, fmt, sf_layout)
    got = fp4.fp4_soft_backward(x.cuda(), q, dy.cuda(), beta).cpu().numpy().astype(np.float64)
    _, s, g = o.quantize(xn, FMT[fmt])
    dyn = dy.float().numpy()
    want = o.soft_backward(xn, s, FMT[fmt], g, dyn, beta)
    xs = o.scaled_inputs(xn, s, FMT[fmt], g)
    err = np.abs(got - want)
    bad = err > grad_tolerance(xs, beta, want, dyn)
    assert not bad.any(), f"{bad.sum()} elements off; worst rel {np.max(err / np.maximum(np.abs(want), 1e-30))}"


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
@pytest.mark.parametrize("beta", BETAS)
def test_soft_forward(fmt, sf_layout, beta):
    x, xn = _input((333, 320), seed=92)
    q = _quantized(x, fmt, sf_layout)
    got = fp4.fp4_soft_forward(x.cuda(), q, beta).cpu().numpy().astype(np.float64)
    _, s, g = o.quantize(xn, FMT[fmt])
    want = o.soft_forward(xn, s, FMT[fmt], g, beta)
    sv = o.block_scales_expanded(s, FMT[fmt], g).astype(np.float64)
    err = np.abs(got - want)
    bad = err > value_tolerance(sv, want)
    assert not bad.any(), f"{bad.sum()} elements off; worst {np.max(err / np.maximum(sv, 1e-38))} block scales"


@pytest.mark.parametrize("x_dtype,dy_dtype", [(torch.float32, torch.float32), (torch.bfloat16, torch.float32),
                                               (torch.float32, torch.bfloat16)])
def test_soft_dtypes_and_pitched_output(x_dtype, dy_dtype):
    x, xn = _input((130, 96), seed=93, dtype=x_dtype)
    rng = np.random.default_rng(94)
    dy = torch.from_numpy(rng.standard_normal((130, 96)).astype(np.float32)).to(dy_dtype)
    q = _quantized(x, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_MMA)
    buf = torch.full((130, 104), 7.0, dtype=torch.float32, device="cuda")
    out = buf[:, :96]
    fp4.fp4_soft_backward(x.cuda(), q, dy.cuda(), 30.0, out=out)
    _, s, g = o.quantize(xn, o.NVFP4)
    dyn = dy.float().numpy()
    want = o.soft_backward(xn, s, o.NVFP4, g, dyn, 30.0)
    xs = o.scaled_inputs(xn, s, o.NVFP4, g)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= grad_tolerance(xs, 30.0, want, dyn))
    assert torch.all(buf[:, 96:] == 7.0)                     # the pitch gap is untouched


def test_soft_large_beta_forward_is_the_dequantized_rtn_value():
    # beta -> inf: s Q_soft(x/s) is the block-scaled RTN dequantization, away
    # from the decision thresholds (an independent route: quantize + dequantize)
    x, xn = _input((256, 256), seed=95)
    q = _quantized(x, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR)
    got = fp4.fp4_soft_forward(x.cuda(), q, 1e5).cpu().numpy()
    deq = fp4.fp4_dequantize(q, out_dtype=torch.float32).cpu().numpy()
    _, s, g = o.quantize(xn, o.NVFP4)
    keep = _dist_to_threshold(o.scaled_inputs(xn, s, o.NVFP4, g)) > 1e-3
    assert np.allclose(got[keep], deq[keep], rtol=1e-6, atol=0)


def test_soft_empty_and_invalid_beta():
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    q = fp4.fp4_quantize(x, fp4.quant_params(fp4.FP4_FMT_NVFP4))
    out = fp4.fp4_soft_backward(x, q, x, 10.0)
    assert out.shape == (0, 64)
    xs, _ = _input((32, 64), seed=96)
    qx = _quantized(xs, fp4.FP4_FMT_NVFP4, fp4.FP4_SF_ROWMAJOR)
    for beta in (0.0, -1.0, float("nan"), 2e6):
        with pytest.raises(RuntimeError):
            fp4.fp4_soft_forward(xs.cuda(), qx, beta)
