"""Pins for the oracle's block-size parameter ("深度学习中的梯度计算基础" §4.2: 16 to 128
elements share one scale) and the relative error of §5.1's table (CPU).

The block size only groups elements: each block's scale comes from its own
amax by the format's rule, and each element is rounded alone.  The brute force
below walks the blocks one by one with the pinned primitives (E8M0 exponent,
E4M3 encoding, E2M1 rounding) and must reproduce quantize() at every size.
"""
import math

import numpy as np
import pytest

import oracle as o


def _brute(x, fmt, block):
    r, c = x.shape
    g = None
    if fmt == o.NVFP4:
        g = np.float32(np.float32(np.abs(x).max()) / np.float32(2688.0))
    codes = np.zeros((r, c), np.uint8)
    scales = np.zeros((r, c // block), np.uint8)
    for i in range(r):
        for j in range(c // block):
            blk = x[i, j * block:(j + 1) * block]
            amax = np.float32(max(abs(float(v)) for v in blk))
            if fmt == o.MXFP4:
                e = int(o.e8m0_exponent(np.array([amax]))[0])
                scales[i, j] = e + 127
                mult = np.float32(2.0 ** -e)
                zero = False
            else:
                sb, mult, zero = o.element_scale_inputs(o.NVFP4, np.array([amax], np.float32), g)
                scales[i, j] = sb[0]
                mult, zero = np.float32(mult[0]), bool(zero[0])
            for k, v in enumerate(blk):
                xs = np.float32(np.float32(v) * mult)
                codes[i, j * block + k] = 0 if zero else o.e2m1_encode_rtn(np.array([xs]))[0]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scales, g


@pytest.mark.parametrize("fmt", [o.MXFP4, o.NVFP4])
@pytest.mark.parametrize("block", [16, 32, 64, 128])
def test_block_sizes_match_a_block_by_block_walk(fmt, block):
    rng = np.random.default_rng(60 + block)
    x = (rng.standard_normal((3, 256)) * np.exp(rng.uniform(-4, 4, (3, 1)))).astype(np.float32)
    x[1, 5] = 40.0                                  # one block with a much larger amax
    x[2, :block] = 0.0                              # an all-zero block
    codes, scales, g = o.quantize(x, fmt, block=block)
    wc, ws, wg = _brute(x, fmt, block)
    assert np.array_equal(scales, ws)
    assert np.array_equal(codes, wc)
    if fmt == o.NVFP4:
        assert np.float32(g) == wg
    # dequantization uses the same grouping
    deq = o.dequantize(codes, scales, fmt, g, block=block).astype(np.float64)
    s = np.repeat(o.block_scale_values(scales, fmt), block, axis=1) * (1.0 if g is None else float(g))
    assert np.allclose(deq, o.e2m1_decode(o.unpack_codes(codes)) * s, rtol=2 ** -23, atol=0)


def test_native_block_is_the_default():
    rng = np.random.default_rng(61)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    for fmt in (o.MXFP4, o.NVFP4):
        a, b = o.quantize(x, fmt), o.quantize(x, fmt, block=o.BLOCK[fmt])
        assert all(np.array_equal(u, v) for u, v in zip(a[:2], b[:2]))


def test_relative_error_closed_forms():
    rng = np.random.default_rng(62)
    x = rng.standard_normal(500)
    assert o.relative_error(x, x) == 0.0
    assert math.isclose(o.relative_error(x, np.zeros_like(x)), 1.0, rel_tol=1e-12)
    assert math.isclose(o.relative_error(x, 1.25 * x), 0.25, rel_tol=1e-12)
    assert math.isclose(o.relative_error(x, -x), 2.0, rel_tol=1e-12)
