"""Pins for the oracle's outlier clamping and compensation (OCC) and the
quantization-quality statistics (CPU).

The MSR write-up (§三) fixes: the threshold is the 99% quantile, only the
largest 1% of values are outliers, they are clamped, and the clamped-away part
is carried by a sparse matrix whose product is computed in high precision.
"""
import math

import numpy as np
import pytest

import oracle as o
from fp4_block_scaled_e8m0_gb300 import inputs


def _count_rule_threshold(a, q):
    # independent formulation: the smallest magnitude t with #{|x| <= t} >= ceil(q n)
    m = np.abs(np.asarray(a, dtype=np.float32)).reshape(-1)
    need = math.ceil(q * m.size)
    for t in np.unique(m):
        if np.count_nonzero(m <= t) >= need:
            return np.float32(t)
    raise AssertionError


@pytest.mark.parametrize("q", [0.5, 0.9, 0.99, 0.999, 1.0])
def test_threshold_is_the_nearest_rank_quantile(q):
    rng = np.random.default_rng(30)
    for shape in [(7, 13), (40, 50), (3, 1)]:
        x = np.round(rng.standard_t(3, shape) * 4).astype(np.float32) / 4     # many ties
        tau = o.occ_threshold(x, q)
        assert tau == _count_rule_threshold(x, q)
        # numpy's type-1 (inverted CDF) quantile is the same order statistic
        assert tau == np.float32(np.quantile(np.abs(x), q, method="inverted_cdf"))


def test_threshold_special_cases():
    x = np.arange(1, 101, dtype=np.float32) * np.where(np.arange(100) % 2, -1, 1)
    assert o.occ_threshold(x, 0.99) == 99.0           # the 99th of 1..100
    assert o.occ_threshold(x, 1.0) == 100.0
    assert o.occ_threshold(x, 0.0) == 1.0             # rank clamps to 1
    # exactly 1% outliers: all of them lie strictly above tau
    a = np.ones(1000, np.float32)
    a[:10] = 500.0
    assert o.occ_threshold(a, 0.99) == 1.0


def test_split_reassembles_exactly():
    rng = np.random.default_rng(31)
    x = inputs.to_bf16(rng.standard_t(3, (64, 96)).astype(np.float32) * 10).float().numpy()
    tau = o.occ_threshold(x)
    xc, dx = o.occ_split(x, tau)
    assert np.array_equal(xc + dx, x)
    assert np.abs(xc).max() <= tau
    outlier = np.abs(x) > tau
    assert np.array_equal(dx != 0, outlier)
    assert outlier.sum() <= x.size - math.ceil(0.99 * x.size)
    r, c, v = o.occ_outliers(x, tau)
    assert np.array_equal(v, dx[r, c]) and len(r) == outlier.sum()
    assert np.all(np.diff(r * 96 + c) > 0)            # row-major order


def _grid_block_matrix(rng, rows, cols):
    """Values of the E2M1 grid with a 4 in every 32-block: MXFP4 scale 2^0, so
    the quantization is exact."""
    g = np.array([0, 0.5, 1, 1.5, 2, 3, 4], np.float32)
    a = rng.choice(g, (rows, cols)) * rng.choice([-1, 1], (rows, cols))
    a[:, ::32] = 4.0
    return a.astype(np.float32)


def test_occ_gemm_is_exact_when_the_clamped_part_quantizes_exactly():
    # X: exact grid values plus 1% huge outliers; clamping at tau = 4 leaves
    # an exactly representable X_c, so Q(X_c) Q(W)^T + dX W^T must be X W^T
    rng = np.random.default_rng(32)
    x = _grid_block_matrix(rng, 64, 64)
    idx = rng.choice(x.size, 40, replace=False)                 # < 1% of 4096
    x.reshape(-1)[idx] = rng.choice([-1000.0, 1000.0, 777.0], 40)
    w = _grid_block_matrix(rng, 48, 64)
    tau = o.occ_threshold(x)
    assert tau == 4.0
    y, bound, _, _ = o.occ_gemm(x, w, o.MXFP4, tau)
    assert np.array_equal(y, x.astype(np.float64) @ w.astype(np.float64).T)
    # and without the compensation the product is wrong (the term matters)
    xc, _ = o.occ_split(x, tau)
    assert not np.allclose(xc.astype(np.float64) @ w.T, y)
    assert np.all(bound >= np.abs(y))


def test_occ_gemm_without_outliers_is_the_plain_gemm():
    rng = np.random.default_rng(33)
    x = rng.standard_normal((32, 64)).astype(np.float32)
    w = rng.standard_normal((16, 64)).astype(np.float32)
    tau = np.float32(np.abs(x).max())
    y, _, _, _ = o.occ_gemm(x, w, o.NVFP4, tau)
    xq, wq = o.quantize(x, o.NVFP4), o.quantize(w, o.NVFP4)
    y0, _ = o.gemm(xq[0], xq[1], wq[0], wq[1], o.NVFP4, xq[2], wq[2])
    assert np.array_equal(y, y0)


def test_error_stats_closed_forms():
    rng = np.random.default_rng(34)
    x = rng.standard_normal(1000)
    s = o.quant_error_stats(x, 2 * x)
    assert math.isclose(s["cos"], 1.0, rel_tol=1e-12)
    assert math.isclose(s["mse"], float(np.mean(x ** 2)), rel_tol=1e-12)
    assert math.isclose(s["snr_db"], 0.0, abs_tol=1e-9)
    assert math.isclose(o.quant_error_stats(x, -x)["cos"], -1.0, rel_tol=1e-12)
    y = np.zeros_like(x)
    y[::2] = 1.0
    z = np.zeros_like(x)
    z[1::2] = 1.0
    assert o.quant_error_stats(y, z)["cos"] == 0.0
    # 10x smaller error power is +10 dB
    e = rng.standard_normal(1000)
    a = o.quant_error_stats(x, x + e)["snr_db"]
    b = o.quant_error_stats(x, x + e / math.sqrt(10))["snr_db"]
    assert math.isclose(b - a, 10.0, rel_tol=1e-9)


def test_reconstruction_without_outliers_is_the_dequantized_value():
    rng = np.random.default_rng(35)
    x = rng.standard_normal((16, 64)).astype(np.float32)
    tau = np.float32(np.abs(x).max())
    rec = o.occ_reconstruction(x, o.NVFP4, tau)
    c, s, g = o.quantize(x, o.NVFP4)
    assert np.array_equal(rec, o.dequantize(c, s, o.NVFP4, g).astype(np.float64))


@pytest.mark.parametrize("fmt", [o.MXFP4, o.NVFP4])
def test_occ_improves_quality_on_hot_channel_activations(fmt):
    # Student-t(3) activations with 1% of the channels x100, as the MSR
    # write-up describes activations (a few huge values, most small): OCC's
    # reconstruction beats direct quantization on all three statistics
    x = inputs.hcp_square(256, 512, 64)["X"].float().numpy()
    tau = o.occ_threshold(x)
    c, s, g = o.quantize(x, fmt)
    direct = o.quant_error_stats(x, o.dequantize(c, s, fmt, g))
    occ = o.quant_error_stats(x, o.occ_reconstruction(x, fmt, tau))
    assert occ["cos"] > direct["cos"] and occ["mse"] < direct["mse"] and occ["snr_db"] > direct["snr_db"]
