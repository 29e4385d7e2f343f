"""Pins for the oracle's block-scaled GEMM and hot-channel compensation (CPU)."""
import numpy as np
import pytest

import oracle as o


def _decode_nibble_by_hand(byte, hi):
    c = (byte >> 4) if hi else (byte & 0xF)
    sign = -1.0 if c & 8 else 1.0
    e, m = (c >> 1) & 3, c & 1
    mag = m * 0.5 if e == 0 else (1.0 + m * 0.5) * 2.0 ** (e - 1)   # E2M1, bias 1
    return sign * mag


@pytest.mark.parametrize("fmt", [o.MXFP4, o.NVFP4])
def test_gemm_matches_triple_loop(fmt):
    rng = np.random.default_rng(21)
    M, N, K = 3, 5, 64
    a = (rng.standard_normal((M, K)) * 2).astype(np.float32)
    b = (rng.standard_normal((N, K)) * 0.1).astype(np.float32)
    ac, asc, ga = o.quantize(a, fmt)
    bc, bsc, gb = o.quantize(b, fmt)
    y, bound = o.gemm(ac, asc, bc, bsc, fmt, ga, gb)
    bsz = o.BLOCK[fmt]

    def scale(sb):
        if fmt == o.MXFP4:
            return 2.0 ** (int(sb) - 127)
        e, m = int(sb) >> 3, int(sb) & 7      # E4M3 by hand
        return (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)

    alpha = 1.0 if fmt == o.MXFP4 else float(ga) * float(gb)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                va = _decode_nibble_by_hand(int(ac[m, k // 2]), k % 2) * scale(asc[m, k // bsz])
                vb = _decode_nibble_by_hand(int(bc[n, k // 2]), k % 2) * scale(bsc[n, k // bsz])
                acc += va * vb
            assert abs(alpha * acc - y[m, n]) <= 1e-12 * max(1.0, bound[m, n])


def test_gemm_closed_form_ones():
    # x = 1 everywhere: MXFP4 scale 2^-2, code 4.0 -> value exactly 1; Y = K
    K = 96
    a = np.ones((4, K), np.float32)
    ac, asc, _ = o.quantize(a, o.MXFP4)
    assert np.all(asc == 125) and np.all(ac == 0x66)
    y, _ = o.gemm(ac, asc, ac, asc, o.MXFP4)
    assert np.all(y == K)


def test_page_error_decomposition_identity():
    # quantized product = exact + first-order + second-order terms (outlier page §3.1)
    rng = np.random.default_rng(22)
    X = rng.standard_normal((8, 64)).astype(np.float32)
    W = (rng.standard_normal((12, 64)) * 0.02).astype(np.float32)
    xc, xs, gx = o.quantize(X, o.NVFP4)
    wc, ws, gw = o.quantize(W, o.NVFP4)
    Xh = o.dequantize(xc, xs, o.NVFP4, gx).astype(np.float64)
    Wh = o.dequantize(wc, ws, o.NVFP4, gw).astype(np.float64)
    dX, dW = Xh - X, Wh - W
    lhs = Xh @ Wh.T
    rhs = X.astype(np.float64) @ W.T + (dX @ W.T + X @ dW.T) + dX @ dW.T
    assert np.allclose(lhs, rhs, atol=1e-12)
    y, bound = o.gemm(xc, xs, wc, ws, o.NVFP4, gx, gw)
    # dequantize rounds each value to fp32 once (2^-24 relative)
    assert np.all(np.abs(y - lhs) <= 2.0 ** -23 * bound)


def _hcp_fixture(fmt, seed=23, M=64, K=128, N=48):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, K)).astype(np.float32)
    hot_true = rng.permutation(K)[:6]
    X[:, hot_true] *= 100
    X = o.bf16_round(X)
    W = o.bf16_round((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    xq = o.quantize(X, fmt)
    wq = o.quantize(W, fmt)
    return X, W, xq, wq, np.sort(hot_true)


@pytest.mark.parametrize("fmt", [o.MXFP4, o.NVFP4])
def test_hcp_order2_equals_plain_definition(fmt):
    X, W, (xc, xs, gx), (wc, ws, gw), _ = _hcp_fixture(fmt)
    h = 12
    hot = o.hcp_select(X, xc, xs, fmt, gx, h)
    y, bound = o.hcp_gemm(X, xc, xs, W, wc, ws, fmt, gx, gw, hot, order=2)
    # plain definition: quantized product on cold channels, exact product on hot ones
    Xh = o.dequantize(xc, xs, fmt, gx).astype(np.float64)
    Wh = o.dequantize(wc, ws, fmt, gw).astype(np.float64)
    mask = np.zeros(X.shape[1], bool)
    mask[hot] = True
    ydef = Xh[:, ~mask] @ Wh[:, ~mask].T + X[:, mask].astype(np.float64) @ W[:, mask].astype(np.float64).T
    # the residual columns are bf16: allow their rounding (2^-8 relative per term)
    tol = 2.0 ** -7 * (np.abs(X[:, mask]) @ np.abs(W[:, mask]).T) + 1e-6 * bound
    assert np.all(np.abs(y - ydef) <= tol)
    # and compensation helps: closer to the unquantized product than plain FP4
    exact = X.astype(np.float64) @ W.astype(np.float64).T
    y0, _ = o.gemm(xc, xs, wc, ws, fmt, gx, gw)
    assert np.abs(y - exact).sum() < np.abs(y0 - exact).sum()


def test_hcp_order1_is_the_literal_concatenation():
    X, W, (xc, xs, gx), (wc, ws, gw), _ = _hcp_fixture(o.NVFP4)
    hot = o.hcp_select(X, xc, xs, o.NVFP4, gx, 8)
    y, bound = o.hcp_gemm(X, xc, xs, W, wc, ws, o.NVFP4, gx, gw, hot, order=1)
    Xh = o.dequantize(xc, xs, o.NVFP4, gx).astype(np.float64)
    Wh = o.dequantize(wc, ws, o.NVFP4, gw).astype(np.float64)
    dW = W[:, hot].astype(np.float64) - Wh[:, hot]
    XH = X[:, hot].astype(np.float64)
    want = Xh @ Wh.T + XH @ dW.T
    tol = 2.0 ** -7 * (np.abs(XH) @ np.abs(dW).T) + 1e-6 * bound
    assert np.all(np.abs(y - want) <= tol)


def test_hcp_with_no_hot_channels_is_the_plain_gemm():
    X, W, (xc, xs, gx), (wc, ws, gw), _ = _hcp_fixture(o.NVFP4)
    y, _ = o.hcp_gemm(X, xc, xs, W, wc, ws, o.NVFP4, gx, gw, np.array([], np.int32))
    y0, _ = o.gemm(xc, xs, wc, ws, o.NVFP4, gx, gw)
    assert np.allclose(y, y0, rtol=1e-12, atol=0)


def test_hcp_select_finds_planted_channels_and_breaks_ties_low():
    X, W, (xc, xs, gx), _, hot_true = _hcp_fixture(o.MXFP4, seed=24)
    hot = o.hcp_select(X, xc, xs, o.MXFP4, None, len(hot_true))
    assert np.array_equal(hot, hot_true)
    assert np.all(np.diff(hot) > 0)
    # all-equal errors: the lowest indices win
    Z = np.zeros((16, 64), np.float32)
    zc, zs, _ = o.quantize(Z, o.MXFP4)
    assert o.hcp_select(Z, zc, zs, o.MXFP4, None, 5).tolist() == [0, 1, 2, 3, 4]


def test_hcp_num_hot_is_ceil_of_nine_percent():
    assert o.hcp_num_hot(4096) == 369
    assert o.hcp_num_hot(100) == 9
    assert o.hcp_num_hot(128) == 12


def _grid_rows(rng, rows, cols):
    # E2M1 grid values with a 4 in every 32-block: MXFP4 scale 2^0, exact quantization
    g = np.array([0, 0.5, 1, 1.5, 2, 3, 4], np.float32)
    a = rng.choice(g, (rows, cols)) * rng.choice([-1, 1], (rows, cols))
    a[:, ::32] = 4.0
    return a.astype(np.float32)


def test_hcp_zeroed_is_exact_when_the_cold_part_quantizes_exactly():
    # X: exact grid values except on the hot channels (arbitrary, huge); W on
    # the grid.  Zeroing H leaves an exactly representable X_0 (every block
    # keeps a 4 at its first column, which is never hot), so the FP4 part is
    # exact and the bf16 columns carry X_H W_H^T exactly: Y = X W^T.
    rng = np.random.default_rng(26)
    X = _grid_rows(rng, 48, 128)
    hot = np.array([3, 40, 77, 100])
    X[:, hot] = o.bf16_round((rng.standard_normal((48, 4)) * 300).astype(np.float32))
    W = _grid_rows(rng, 40, 128)
    y, bound, _, _ = o.hcp_zeroed_gemm(X, W, o.MXFP4, hot)
    assert np.array_equal(y, X.astype(np.float64) @ W.astype(np.float64).T)
    assert np.all(bound >= np.abs(y))
    # the plain FP4 product is not exact: the hot values inflate their blocks
    xq, wq = o.quantize(X, o.MXFP4), o.quantize(W, o.MXFP4)
    y0, _ = o.gemm(xq[0], xq[1], wq[0], wq[1], o.MXFP4)
    assert not np.allclose(y0, y)


def test_hcp_zeroed_without_hot_channels_is_the_plain_gemm():
    X, W, (xc, xs, gx), (wc, ws, gw), _ = _hcp_fixture(o.NVFP4)
    y, _, _, _ = o.hcp_zeroed_gemm(X, W, o.NVFP4, np.array([], np.int64))
    y0, _ = o.gemm(xc, xs, wc, ws, o.NVFP4, gx, gw)
    assert np.array_equal(y, y0)


@pytest.mark.parametrize("fmt", [o.MXFP4, o.NVFP4])
def test_hcp_zeroed_shrinks_the_hot_blocks_and_the_error(fmt):
    X, W, (xc, xs, gx), (wc, ws, gw), hot_true = _hcp_fixture(fmt, seed=27)
    hot = o.hcp_select(X, xc, xs, fmt, gx, len(hot_true))
    y, _, (zc, zs, zg), _ = o.hcp_zeroed_gemm(X, W, fmt, hot)
    # block scales (values, with the tensor scale) no larger than before, and
    # much smaller, in total, in the blocks that held a hot channel
    s_old = o.block_scales_expanded(xs, fmt, gx)
    s_new = o.block_scales_expanded(zs, fmt, zg)
    assert np.all(s_new <= s_old * (1 + 2 ** -3))      # E4M3 rounding under a new tensor scale
    assert s_new[:, hot].sum() < 0.1 * s_old[:, hot].sum()
    exact = X.astype(np.float64) @ W.astype(np.float64).T
    y0, _ = o.gemm(xc, xs, wc, ws, fmt, gx, gw)
    assert np.abs(y - exact).sum() < 0.5 * np.abs(y0 - exact).sum()


def test_e4m3_rows_exact_on_representable_rows():
    # rows of E4M3 values times 2^k whose largest magnitude is 448 * 2^k: the
    # scale is exactly 2^k and every value comes back unchanged
    rng = np.random.default_rng(28)
    table = o.E4M3_VALUES[:127]
    rows = []
    for k in (-20, -3, 0, 5):
        r = rng.choice(table, 40) * rng.choice([-1, 1], 40)
        r[7] = -448.0
        rows.append(r * 2.0 ** k)
    v = np.array(rows, np.float32)
    vals, s = o.e4m3_rows(v)
    assert np.array_equal(s, np.float32([2.0 ** k for k in (-20, -3, 0, 5)]))
    assert np.array_equal(vals * s.astype(np.float64)[:, None], v.astype(np.float64))


def test_e4m3_rows_relative_precision_and_zero_rows():
    rng = np.random.default_rng(29)
    v = (rng.standard_normal((8, 64)) * np.exp(rng.uniform(-5, 5, (8, 1)))).astype(np.float32)
    v[3] = 0.0
    vals, s = o.e4m3_rows(v)
    back = vals * s.astype(np.float64)[:, None]
    assert np.all(back[3] == 0) and s[3] == 0
    # normal range of the row (>= 2^-6 s): within half an E4M3 ulp (2^-4 relative)
    normal = (np.abs(v) >= (2.0 ** -6) * s[:, None]) & (v != 0)
    rel = np.abs(back - v)[normal] / np.abs(v)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-12


@pytest.mark.parametrize("order", [0, 1, 2])
def test_hcp_fp8_tail_is_the_bf16_tail_within_e4m3_precision(order):
    X, W, (xc, xs, gx), (wc, ws, gw), _ = _hcp_fixture(o.NVFP4, seed=30)
    hot = o.hcp_select(X, xc, xs, o.NVFP4, gx, 10)
    if order == 0:
        xc, xs, gx = o.quantize(o.hcp_zero_columns(X, hot), o.NVFP4)
        y16, _, _, _ = o.hcp_zeroed_gemm(X, W, o.NVFP4, hot)
    else:
        y16, _ = o.hcp_gemm(X, xc, xs, W, wc, ws, o.NVFP4, gx, gw, hot, order)
    y8, _ = o.hcp_gemm_fp8(X, xc, xs, W, wc, ws, o.NVFP4, gx, gw, hot, order)
    a, b = o.hcp_fp8_columns(X, xc, xs, W, wc, ws, o.NVFP4, gx, gw, hot, order)
    mag = np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64)).T
    # each product term: E4M3 (2^-4 each, subnormal tail small) and bf16 (2^-8 each) roundings
    assert np.all(np.abs(y8 - y16) <= 0.15 * mag + 1e-6 * np.abs(y16))
    # and the tail matters: dropping it moves Y by much more
    y0, _ = o.gemm(xc, xs, wc, ws, o.NVFP4, gx, gw)
    assert np.abs(y0 - y16).sum() > 5 * np.abs(y8 - y16).sum()
