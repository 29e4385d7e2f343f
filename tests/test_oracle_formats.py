"""Pins for the oracle's number formats and quantizer (CPU only).

Each test checks the oracle against something other than itself: values printed
or fixed by the pages, hand-derived fixtures, an independent formulation, a
library routine (torch's fp8 / bf16 casts) or brute force on tiny inputs.
"""
import numpy as np
import pytest
import torch

import oracle as o
from conftest import golden


def test_e2m1_grid_and_range():
    # E2M1: 16 codes, values 0, +-0.5 ... +-6 (outlier page §1.1: range [-6, 6]).
    vals = o.e2m1_decode(np.arange(16))
    assert sorted(set(np.abs(vals))) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert vals.max() == 6.0 and vals.min() == -6.0
    assert np.all(vals[8:] == -vals[:8])


def test_e2m1_rtn_golden_points():
    rows = golden("e2m1_rtn_points.txt")
    xs = np.array([float(r[0]) for r in rows], dtype=np.float32)
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint8)
    got = o.e2m1_encode_rtn(xs)
    assert np.array_equal(got, want), list(zip(xs, got, want))


def _e2m1_rtn_ieee(xs):
    """Independent formulation: round |x| to 1 mantissa bit per binade, half-even
    on the *value* (np.round), subnormal step 0.5 below 1, saturate at 6."""
    a = np.abs(xs.astype(np.float64))
    v = np.where(a < 2.0, np.round(a * 2.0) / 2.0,
                 np.where(a < 4.0, np.round(a), np.round(a / 2.0) * 2.0))
    v = np.minimum(v, 6.0)
    lut = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    mag = np.vectorize(lut.__getitem__)(v).astype(np.uint8)
    return (np.signbit(xs).astype(np.uint8) << 3) | mag


@pytest.mark.parametrize("mult", [1.0, 4.0, 0.03125, 1.0 / 3.0])
def test_e2m1_rtn_all_bf16_patterns(mult):
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    xs = (x * np.float32(mult)).astype(np.float32)
    xs = xs[np.isfinite(xs)]
    assert np.array_equal(o.e2m1_encode_rtn(xs), _e2m1_rtn_ieee(xs))


def test_e2m1_idempotent_on_grid():
    vals = o.e2m1_decode(np.arange(16)).astype(np.float32)
    assert np.array_equal(o.e2m1_encode_rtn(vals), np.arange(16, dtype=np.uint8))


def test_e4m3_against_torch():
    rng = np.random.default_rng(7)
    table = o.E4M3_VALUES[:127]
    mids = (table[1:] + table[:-1]) / 2
    t = np.concatenate([table, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
                        rng.uniform(0, 448, 20000), np.exp(rng.uniform(-12, 6, 20000)),
                        [0.0, 448.0, 2.0 ** -10, 2.0 ** -9.5]]).astype(np.float32)
    t = t[(t >= 0) & (t <= 448)]
    want = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.e4m3_encode_rn_satfinite(t), want)
    # satfinite: above the largest finite value clamps to 448 (byte 0x7E)
    assert np.all(o.e4m3_encode_rn_satfinite(np.float32([449.0, 500.0, 1e6])) == 0x7E)
    assert np.allclose(o.e4m3_decode(np.arange(127)), table)


def _num(v: str) -> float:
    return float.fromhex(v) if "p" in v else float(v)


def test_e8m0_golden_points():
    rows = golden("e8m0_scale_points.txt")
    amax = np.array([_num(r[0]) for r in rows], dtype=np.float32)
    hexpts = np.array([_num(r[0]) for r in rows if "p" in r[0]])
    assert np.array_equal(hexpts.astype(np.float32).astype(np.float64), hexpts)   # the hex points are fp32 values
    want = np.array([int(r[1]) for r in rows])
    assert np.array_equal(o.e8m0_exponent(amax) + 127, want)


def test_mxfp4_tiny_blocks_golden():
    """Blocks of bf16-subnormal and tiny values (hand-derived codes and bytes):
    the exponent clamp at -127, the true exponent of subnormal amax, and no
    flush of subnormal elements to zero before the scaling."""
    rows = golden("mxfp4_tiny_blocks.txt")
    blocks = sorted({r[0] for r in rows})
    x = np.zeros((len(blocks), 32), np.float32)
    want_codes = np.zeros((len(blocks), 32), np.uint8)
    want_bytes = np.zeros((len(blocks), 1), np.uint8)
    for r in rows:
        b = blocks.index(r[0])
        if r[1] == "scale":
            want_bytes[b, 0] = int(r[2])
        else:
            x[b, int(r[1])] = _num(r[2])
            want_codes[b, int(r[1])] = int(r[3])
    assert np.array_equal(o.bf16_round(x).view(np.uint32), x.view(np.uint32))   # bf16 values, as the fixture says
    codes, scales, _ = o.quantize(x, o.MXFP4)
    assert np.array_equal(scales, want_bytes)
    assert np.array_equal(o.unpack_codes(codes), want_codes)
    # dequantized values: code value * 2^(byte - 127), exact even when subnormal in fp32
    deq = o.dequantize(codes, scales, o.MXFP4)
    want_deq = o.e2m1_decode(want_codes) * np.ldexp(1.0, want_bytes.astype(np.int64) - 127)
    assert np.array_equal(deq.astype(np.float64), want_deq)


def test_e8m0_amax_over_scale_in_4_8():
    rng = np.random.default_rng(3)
    amax = np.exp(rng.uniform(-80, 80, 100000)).astype(np.float32)
    e = o.e8m0_exponent(amax)
    ratio = amax.astype(np.float64) / np.ldexp(1.0, e)
    assert np.all((ratio >= 4.0) & (ratio < 8.0))


def test_bf16_round_against_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(100000) * 10 ** rng.uniform(-30, 30, 100000),
                        (np.arange(1 << 16, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    x = x.astype(np.float32)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = o.bf16_round(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def _brute_force_nearest_code(x, s):
    """Among all 16 codes (value cv * s) the one nearest to x; ties to even code."""
    cands = o.e2m1_decode(np.arange(16)) * s
    d = np.abs(x - cands)
    best = d.min()
    idx = [c for c in range(16) if d[c] == best]
    # +-0 are both nearest for tiny x: prefer the one with x's sign
    idx = [c for c in idx if (c >= 8) == bool(np.signbit(x))] or idx
    even = [c for c in idx if c % 2 == 0]
    return (even or idx)[0]


@pytest.mark.parametrize("fmt", [o.MXFP4, o.NVFP4])
def test_quantize_rtn_is_nearest_by_brute_force(fmt):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((3, 64)) * np.array([[1.0], [37.0], [1e-3]])).astype(np.float32)
    x[0, 5] = 0.0
    x[1, 3] = -0.0
    codes, scales, g = o.quantize(x, fmt)
    c = o.unpack_codes(codes)
    bsz = o.BLOCK[fmt]
    for r in range(x.shape[0]):
        for j in range(x.shape[1]):
            sb = scales[r, j // bsz]
            s = 2.0 ** (int(sb) - 127) if fmt == o.MXFP4 else float(o.e4m3_decode(sb)) * float(g)
            # the value the oracle scaled (fp32 x * (1/s)) is what RTN rounds
            assert c[r, j] == _brute_force_nearest_code(float(x[r, j]) / s, 1.0), (r, j)


def test_nvfp4_scale_sequence_invariants():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((32, 256)) * 3).astype(np.float32)
    x[:, 17] *= 100
    codes, scales, g = o.quantize(x, o.NVFP4)
    amax_t = np.abs(x).max()
    assert abs(float(g) * 2688 - amax_t) <= 1e-6 * amax_t
    amax_b = np.abs(x).reshape(32, 16, 16).max(axis=2)
    dec = o.e4m3_decode(scales) * float(g) * 6
    # E4M3 keeps 3 mantissa bits: decoded scale within 2^-4 relative of amax_b/6
    ok = amax_b > 2.0 ** -6 * 6 * float(g)
    assert np.all(np.abs(dec[ok] - amax_b[ok]) <= 2.0 ** -4 * amax_b[ok])
    # the block max lands on or next to the top of the grid
    xs_max = amax_b / (o.e4m3_decode(scales) * float(g))
    assert np.all((xs_max[ok] > 5.0) & (xs_max[ok] < 6.5))


def test_nvfp4_zero_tensor_gives_zero_scales_and_codes():
    x = np.zeros((16, 32), dtype=np.float32)
    x[3, 4] = -0.0
    codes, scales, g = o.quantize(x, o.NVFP4)
    assert g == 0 and not codes.any() and not scales.any()


def test_2d_scale_is_max_of_row_scales():
    # one scale per 16x16 tile (outlier page §4.1 "2D scaling", §4.2 block_16x16)
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((48, 64)) * rng.uniform(0.1, 10, (48, 1))).astype(np.float32)
    _, s1, g1 = o.quantize(x, o.NVFP4, scaling="1d")
    _, s2, g2 = o.quantize(x, o.NVFP4, scaling="2d")
    assert g1 == g2
    want = s1.reshape(3, 16, 4).max(axis=1)       # E4M3 encoding is monotonic
    assert np.array_equal(s2[::16], want)
    assert np.array_equal(s2, np.repeat(want, 16, axis=0))


def test_transpose_and_rht_are_compositions():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((64, 32)).astype(np.float32)
    a = o.quantize(x, o.NVFP4, transpose=True)
    b = o.quantize(np.ascontiguousarray(x.T), o.NVFP4)
    assert all(np.array_equal(p, q) for p, q in zip(a[:2], b[:2])) and a[2] == b[2]
    c = o.quantize(x, o.MXFP4, rht=True, rht_seed=9)
    d = o.quantize(o.rht16(x, 1, 9), o.MXFP4)
    assert all(np.array_equal(p, q) for p, q in zip(c[:2], d[:2]))


def test_mxfp4_quantize_is_idempotent():
    # Q(Q(x)) = Q(x): a block's dequantized max keeps the same E8M0 exponent
    rng = np.random.default_rng(15)
    x = (rng.standard_normal((8, 64)) * 10 ** rng.uniform(-3, 3, (8, 1))).astype(np.float32)
    codes, scales, _ = o.quantize(x, o.MXFP4)
    xh = o.dequantize(codes, scales, o.MXFP4)
    codes2, scales2, _ = o.quantize(xh, o.MXFP4)
    assert np.array_equal(codes2, codes) and np.array_equal(scales2, scales)
    assert np.array_equal(o.dequantize(codes2, scales2, o.MXFP4), xh)
