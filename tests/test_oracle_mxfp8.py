"""Pins of the oracle's MXFP8 extra columns (single-kernel hot-channel tail):
the block exponent against a brute-force search and hand-derived points, the
element rounding against torch's float8_e4m3fn cast, and the product against
the bf16-tail oracle on columns that MXFP8 represents exactly."""
import numpy as np
import pytest
import torch

import oracle as o
from conftest import golden


def _brute_exponent(a: float) -> int:
    """smallest e in [-127, 127] with a <= 448 * 2^e (exact fp64), -127 below."""
    for e in range(-127, 128):
        if a <= 448.0 * 2.0 ** e:
            return e
    raise AssertionError("no exponent")


def test_mxfp8_exponent_brute_force():
    rng = np.random.default_rng(0)
    a = np.concatenate([
        np.exp2(rng.uniform(-149, 127, 4000)),
        np.exp2(np.arange(-149, 128, dtype=np.float64)),            # powers of two
        0.875 * np.exp2(np.arange(-120, 120, dtype=np.float64)),    # the 7/8 boundary
    ]).astype(np.float32)
    a = np.concatenate([a, np.nextafter(a, np.float32(np.inf)), np.nextafter(a, np.float32(0))])
    a = a[np.isfinite(a)]
    got = o.mxfp8_exponent(a)
    want = np.array([_brute_exponent(float(v)) for v in a])
    assert np.array_equal(got, want)
    assert o.mxfp8_exponent(np.float32(0.0)) == -127


def test_mxfp8_exponent_golden():
    rows = golden("mxfp8_scale_points.txt")
    for r in rows:
        a = float.fromhex(r[0])
        assert o.mxfp8_exponent(np.float32(a)) == int(r[1]), r


def test_mxfp8_elements_match_torch_e4m3_cast():
    rng = np.random.default_rng(1)
    v = (rng.standard_t(3, (64, 256)) * np.exp2(rng.uniform(-30, 30, (64, 1)))).astype(np.float32)
    codes, e = o.mxfp8_quantize_rows(v)
    t = (np.abs(v).reshape(64, 8, 32).astype(np.float64) * np.exp2(-e.astype(np.float64))[:, :, None]).astype(np.float32)
    assert t.max() <= 448.0                                   # no element saturates
    ref = torch.from_numpy(t.reshape(64, 256)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes & 0x7F, ref)
    assert np.array_equal(codes >> 7, np.signbit(v).astype(np.uint8))
    # every block's scaled amax lies in (224, 448] (the smallest such power of
    # two), and its rounded value in [224, 448]
    tmax = t.max(axis=2)
    assert np.all((tmax > 224) & (tmax <= 448))
    top = np.abs(o.mxfp8_values(codes, e).reshape(64, 8, 32)).max(axis=2) / np.exp2(e)
    assert np.all((top >= 224) & (top <= 448))


def _e4m3_grid_rows(rng, rows, cols, k):
    """values on the E4M3 grid times 2^k (per row), each 32-block holding +-448 * 2^k."""
    grid = o.E4M3_VALUES[:127]
    v = rng.choice(grid, (rows, cols)) * np.where(rng.random((rows, cols)) < 0.5, -1.0, 1.0)
    v[:, ::32] = 448.0
    return (v * np.exp2(k)[:, None]).astype(np.float32)


def test_mxfp8_tail_exact_on_representable_columns():
    """MXFP4, order 0: A = X_H, B = W_H (alpha = 1).  With X_H and W_H on the E4M3
    grid and every block's amax 448 * 2^k, the MXFP8 columns are exact, and the
    product equals the bf16-tail oracle's (the values are bf16-exact too)."""
    rng = np.random.default_rng(2)
    M, N, K, h = 40, 24, 256, 64
    hot = np.sort(rng.permutation(K)[:h])
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x[:, hot] = _e4m3_grid_rows(rng, M, h, rng.integers(-6, 4, M))
    w[:, hot] = _e4m3_grid_rows(rng, N, h, rng.integers(-12, -4, N))
    xb = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    wb = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    assert np.array_equal(xb[:, hot], x[:, hot]) and np.array_equal(wb[:, hot], w[:, hot])
    xz = o.hcp_zero_columns(xb, hot)
    cx, sx, gx = o.quantize(xz, o.MXFP4)
    cw, sw, gw = o.quantize(wb, o.MXFP4)
    y8, _ = o.hcp_gemm_mxfp8(xb, cx, sx, wb, cw, sw, o.MXFP4, gx, gw, hot, order=0)
    yz = o.hcp_zeroed_gemm(xb, wb, o.MXFP4, hot)[0]
    # the same terms summed in fp64 (the two oracles group the sums alike up to BLAS order)
    assert np.allclose(y8, yz, rtol=1e-12, atol=0.0)
    a, b = o.hcp_mxfp8_columns(xb, cx, sx, wb, cw, sw, o.MXFP4, gx, gw, hot, order=0)
    assert np.array_equal(o.mxfp8_values(*o.mxfp8_quantize_rows(a)), a.astype(np.float64))


@pytest.mark.parametrize("order", [0, 1, 2])
@pytest.mark.parametrize("fmt", [o.MXFP4, o.NVFP4])
def test_mxfp8_tail_within_e4m3_precision(order, fmt):
    """The MXFP8 tail differs from the unrounded fp32 columns' product by at most
    E4M3's relative half-step (2^-4) on each factor: |A8 B8 - A B| <= sum |a||b| (2^-3 + 2^-8)."""
    rng = np.random.default_rng(3 + order)
    M, N, K, h = 48, 40, 512, 41
    x = rng.standard_t(3, (M, K)).astype(np.float32)
    x[:, rng.permutation(K)[:8]] *= 100
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    wb = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    cx, sx, gx = o.quantize(xb, fmt)
    cw, sw, gw = o.quantize(wb, fmt)
    hot = o.hcp_select(xb, cx, sx, fmt, gx, h)
    if order == 0:
        cx, sx, gx = o.quantize(o.hcp_zero_columns(xb, hot), fmt)
    a, b = o.hcp_mxfp8_columns(xb, cx, sx, wb, cw, sw, fmt, gx, gw, hot, order)
    A8 = o.mxfp8_values(*o.mxfp8_quantize_rows(a))
    B8 = o.mxfp8_values(*o.mxfp8_quantize_rows(b))
    exact = a.astype(np.float64) @ b.astype(np.float64).T
    bound = np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64).T
    assert np.all(np.abs(A8 @ B8.T - exact) <= bound * (2.0 ** -3 + 2.0 ** -8) + 1e-300)
    # and the part layout: each part starts on a 32-column boundary
    kp = -(-h // 32) * 32
    assert a.shape[1] == (2 if order == 2 else 1) * kp
    assert not np.any(a[:, h:kp])
