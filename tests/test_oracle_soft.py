"""Pins for the oracle's sigmoid-smoothed quantizer Q_soft and its derivative (CPU).

The page ("深度学习中的梯度计算基础", §3.2) fixes three properties: Q_soft tends to
the standard quantizer as beta grows, it is differentiable everywhere, and its
derivative is beta sum v_i sigma (1 - sigma).  The pins below check the oracle
against those, against the independent RTN encoder, and against closed forms.
"""
import numpy as np
import pytest

import oracle as o


def _thresholds():
    return o.soft_grid()[1]


def test_soft_grid_is_the_signed_e2m1_grid():
    q, c, v = o.soft_grid()
    # the 15 distinct values of the 16 codes, decoded by the format's own table
    want = np.unique(o.e2m1_decode(np.arange(16, dtype=np.uint8)))
    assert np.array_equal(q, want)
    assert np.all((q[:-1] < c) & (c < q[1:]))
    assert v.sum() == 12.0 and np.all(v > 0)


def _away_from_thresholds(xs, gap):
    d = np.abs(np.asarray(xs, dtype=np.float64)[..., None] - _thresholds()).min(axis=-1)
    return d > gap


def test_soft_tends_to_round_to_nearest():
    # beta -> inf: Q_soft is RTN onto the E2M1 grid, saturating at +-6
    rng = np.random.default_rng(21)
    xs = rng.uniform(-9.0, 9.0, 20000).astype(np.float32)
    keep = _away_from_thresholds(xs, 0.01)
    xs = xs[keep]
    rtn = o.e2m1_decode(o.e2m1_encode_rtn(xs))
    got = o.soft_quantize_scaled(xs, beta=1e4)
    assert np.allclose(got, rtn, rtol=0, atol=1e-12)
    # and far from it for a small beta: the smoothing is real
    assert np.abs(o.soft_quantize_scaled(xs, beta=2.0) - rtn).max() > 0.1


def test_soft_midpoint_value_and_peak_slope_at_each_threshold():
    q, c, v = o.soft_grid()
    beta = 1e4
    # at c_i only sigma(0) = 1/2 is undecided: the value is halfway up the step
    assert np.allclose(o.soft_quantize_scaled(c, beta), 0.5 * (q[:-1] + q[1:]), atol=1e-12)
    # sigma (1 - sigma) peaks at 1/4
    assert np.allclose(o.soft_derivative(c, beta), beta * v / 4.0, rtol=1e-12)


@pytest.mark.parametrize("beta", [1.0, 10.0, 40.0, 100.0])
def test_soft_derivative_is_the_slope_of_q_soft(beta):
    rng = np.random.default_rng(int(beta))
    xs = rng.uniform(-7.0, 7.0, 4000)
    h = 1e-5 / beta
    fd = (o.soft_quantize_scaled(xs + h, beta) - o.soft_quantize_scaled(xs - h, beta)) / (2 * h)
    got = o.soft_derivative(xs, beta)
    # central differences: error O(h^2 Q''') plus cancellation ~1e-16 / h
    assert np.allclose(got, fd, rtol=1e-6, atol=1e-9 * beta)


@pytest.mark.parametrize("beta", [1.0, 10.0, 100.0])
def test_soft_derivative_integrates_to_the_grid_span(beta):
    # integral over the line = Q(+inf) - Q(-inf) = 6 - (-6)
    lim = 6.0 + 40.0 / beta
    n = 2_000_000
    h = 2 * lim / n
    mid = -lim + (np.arange(n) + 0.5) * h
    assert abs(o.soft_derivative(mid, beta).sum() * h - 12.0) < 1e-6


def test_soft_small_beta_is_linear():
    # sigma(z) = 1/2 + z/4 + O(z^3) and sum v_i c_i = (q_14^2 - q_0^2)/2 = 0, so
    # Q_soft(x) = 3 beta x + O(beta^3) and Q_soft'(x) = 3 beta + O(beta^3)
    beta = 1e-5
    xs = np.linspace(-7, 7, 57)
    assert np.allclose(o.soft_quantize_scaled(xs, beta), 3 * beta * xs, rtol=1e-6, atol=1e-15)
    assert np.allclose(o.soft_derivative(xs, beta), 3 * beta, rtol=1e-6)


def test_soft_is_odd_with_even_derivative():
    xs = np.linspace(-8, 8, 1601)
    for beta in (1.0, 7.0, 60.0):
        assert np.allclose(o.soft_quantize_scaled(-xs, beta), -o.soft_quantize_scaled(xs, beta),
                           rtol=0, atol=1e-13)
        assert np.allclose(o.soft_derivative(-xs, beta), o.soft_derivative(xs, beta), rtol=1e-13)
        d = o.soft_derivative(xs, beta)
        assert np.all(d > 0)
        assert np.all(np.abs(o.soft_quantize_scaled(xs, beta)) <= 6.0)


def test_soft_derivative_tail_keeps_relative_precision():
    # xs = 4.25 is 0.75 from both neighbouring thresholds (3.5 and 5, steps 1
    # and 2); every other threshold is >= 1.5 further.  With beta = 100 the two
    # terms are beta v e^-75 / (1 + e^-75)^2 each: far below 1 - sigma's fp64
    # resolution, so a naive sigma (1 - sigma) would give 0
    beta = 100.0
    e = np.exp(-75.0)
    want = beta * (1.0 + 2.0) * e / (1.0 + e) ** 2
    assert np.isclose(o.soft_derivative(np.array([4.25]), beta)[0], want, rtol=1e-12)


def test_soft_forward_backward_use_the_quantizer_scaling():
    rng = np.random.default_rng(22)
    x = (rng.standard_normal((16, 64)) * 3).astype(np.float32)
    dy = rng.standard_normal((16, 64)).astype(np.float32)
    for fmt in (o.MXFP4, o.NVFP4):
        codes, scales, g = o.quantize(x, fmt)
        xs = o.scaled_inputs(x, scales, fmt, g)
        keep = _away_from_thresholds(xs, 1e-3)
        # large beta: the smoothed forward is the block-scaled RTN dequantization
        y = o.soft_forward(x, scales, fmt, g, beta=1e6)
        deq = o.dequantize(codes, scales, fmt, g).astype(np.float64)
        assert np.allclose(y[keep], deq[keep], rtol=1e-6, atol=0)
        dx = o.soft_backward(x, scales, fmt, g, dy, beta=10.0)
        assert np.allclose(dx, dy * o.soft_derivative(xs.astype(np.float64), 10.0))
