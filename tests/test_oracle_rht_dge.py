"""Pins for the oracle's 16-point random Hadamard transform and the DGE (CPU)."""
import numpy as np
import pytest
import scipy.linalg

import oracle as o
from conftest import golden


def test_butterfly_equals_sylvester_hadamard():
    # y = 1/4 H16 x with all signs +1: each basis vector maps to a column of H16
    eye = np.eye(16, dtype=np.float32)
    y = o.rht16_chunks(eye, np.ones(16, dtype=np.float32))      # row j = transform of e_j
    H = scipy.linalg.hadamard(16).astype(np.float64)
    assert np.array_equal(y.astype(np.float64), 0.25 * H.T)
    assert np.array_equal(H @ H.T, 16 * np.eye(16))


def test_rht_signs_are_rademacher_from_philox():
    s = o.rht16_signs(2)
    assert set(s) <= {-1.0, 1.0}
    w0 = int(o.philox4x32_10((0, 0, 0, 0), (2, 0))[0])
    assert [int(v < 0) for v in s] == [(w0 >> j) & 1 for j in range(16)]
    assert not np.array_equal(o.rht16_signs(2), o.rht16_signs(3))


def test_rht_is_orthogonal():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    for axis in (0, 1):
        y = o.rht16(x, axis, seed=2)
        xs = x.reshape(64, 8, 16) if axis == 1 else x.T.reshape(128, 4, 16)
        ys = y.reshape(64, 8, 16) if axis == 1 else y.T.reshape(128, 4, 16)
        n0 = np.linalg.norm(xs.astype(np.float64), axis=-1)
        n1 = np.linalg.norm(ys.astype(np.float64), axis=-1)
        assert np.allclose(n0, n1, rtol=1e-6)
    # inverse: x = D (1/4 H) y  since (1/4 H D)^T (1/4 H D) = I
    y = o.rht16(x, 1, seed=5)
    back = o.rht16_chunks(y.reshape(64, 8, 16), np.ones(16, np.float32)) * o.rht16_signs(5)
    assert np.allclose(back.reshape(64, 128), x, atol=1e-5)


def test_rht_preserves_products_along_the_reduction_axis():
    # (A R)(B R)^T = A B^T when both operands get the same R along K
    rng = np.random.default_rng(6)
    A = rng.standard_normal((24, 64)).astype(np.float32)
    B = rng.standard_normal((40, 64)).astype(np.float32)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    got = o.rht16(A, 1, 2).astype(np.float64) @ o.rht16(B, 1, 2).astype(np.float64).T
    assert np.allclose(got, ref, atol=1e-4)
    bad = o.rht16(A, 1, 2).astype(np.float64) @ o.rht16(B, 1, 3).astype(np.float64).T
    assert not np.allclose(bad, ref, atol=1e-2)


def test_dge_golden_points():
    rows = golden("dge_points.txt")
    xs = np.array([float(r[0]) for r in rows], dtype=np.float32)
    want = np.array([float(r[1]) for r in rows])
    got = o.dge_derivative(xs, k=5.0, clamp=3.0)
    assert np.allclose(got, want, rtol=1e-12, atol=0)


def _f_page(x, d, k):
    """The pages' f(x) = d/2 (1 + sign(2x/d - 1) |2x/d - 1|^(1/k)) on [0, d)."""
    t = 2.0 * x / d - 1.0
    return d / 2.0 * (1.0 + np.sign(t) * np.abs(t) ** (1.0 / k))


@pytest.mark.parametrize("k", [3.0, 5.0, 9.0])
def test_dge_is_derivative_of_page_formula(k):
    grid = o.E2M1_GRID
    rng = np.random.default_rng(8)
    for i in range(7):
        lo, d = grid[i], grid[i + 1] - grid[i]
        # stay off the clamp region and the interval ends
        t = rng.uniform(0.15, 0.95, 40) * rng.choice([-1, 1], 40)
        xs = lo + (t + 1.0) * d / 2.0
        h = 1e-6 * d
        fd = (_f_page(xs - lo + h, d, k) - _f_page(xs - lo - h, d, k)) / (2 * h)
        got = o.dge_derivative(xs.astype(np.float32).astype(np.float64), k, clamp=np.inf)
        # xs rounded to fp32 in the oracle: compare at that point
        xs32 = xs.astype(np.float32).astype(np.float64)
        fd32 = (_f_page(xs32 - lo + h, d, k) - _f_page(xs32 - lo - h, d, k)) / (2 * h)
        assert np.allclose(got, fd32, rtol=1e-5), (i, k)


def test_dge_integral_over_each_interval():
    # unclamped: the integral of f' over an interval is the interval width d
    # (f rises from 0 to d); with the clamp at c it is d (c u_c + 1 - u_c^(1/k))
    k, c = 5.0, 3.0
    uc = (1.0 / (c * k)) ** (k / (k - 1.0))
    want_frac = c * uc + 1.0 - uc ** (1.0 / k)
    grid = o.E2M1_GRID
    n = 400000
    for i in range(7):
        lo, d = grid[i], grid[i + 1] - grid[i]
        mid = lo + (np.arange(n) + 0.5) * d / n
        integral = o.dge_derivative(mid, k, c).sum() * d / n
        assert abs(integral - d * want_frac) < 1e-4 * d


def test_dge_continuous_at_grid_points_and_outside():
    grid = o.E2M1_GRID[1:7]
    left = o.dge_derivative(np.nextafter(grid.astype(np.float32), np.float32(0)), 5.0, 3.0)
    right = o.dge_derivative(grid.astype(np.float32), 5.0, 3.0)
    assert np.allclose(left, 0.2, rtol=1e-5) and np.allclose(right, 0.2, rtol=0)
    assert o.dge_derivative(np.float32([6.0, -7.0]), 5.0, 3.0, outside=0.0).tolist() == [0.0, 0.0]


def test_dge_backward_uses_the_quantizer_scaling():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 64)).astype(np.float32)
    dy = rng.standard_normal((16, 64)).astype(np.float32)
    for fmt in (o.MXFP4, o.NVFP4):
        codes, scales, g = o.quantize(x, fmt)
        dx = o.dge_backward(x, scales, fmt, g, dy)
        # the derivative is taken at x/s: its grid interval is the one the code sits in
        xs = o.scaled_inputs(x, scales, fmt, g).astype(np.float64)
        assert np.allclose(dx, dy * o.dge_derivative(xs, 5.0, 3.0))
        cv = o.e2m1_decode(o.unpack_codes(codes))
        inside = np.abs(xs) <= 6.0
        assert np.all(np.abs(cv - xs)[inside] <= 1.0)          # half of the widest step
        assert np.all(np.abs(cv[~inside]) == 6.0)
