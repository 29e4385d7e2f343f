"""Plain CPU oracle for block-scaled FP4 quantization and the GEMMs that consume it.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

Every function is written to be checked by eye against the pages it follows.
The pages are cited by short names:

* [grad]    aicoding.csdn.net, "深度学习中的梯度计算基础" (gradient estimators for
            quantization, MXFP4 block size)
* [lowprec] framerc.cn, "低精度训练技术概述" (low-precision training survey:
            E4M3 / E8M0 / MXFP4 / NVFP4 formats, stochastic-rounding snippet)
* [outlier] devpress.csdn.net, "大模型4位训练中的异常值动态分析与优化实践"
            (NVFP4 outliers, hot-channel compensation, the CHON recipe)
* [msr]     lsdiaocha.cn, news write-up of the MSR FP4-training paper (E2M1,
            differentiable gradient estimator, outlier clamping)

Arithmetic: fp64 where the result is a real number the method defines (GEMM
sums, the DGE derivative, hot-channel errors).  Where floating point decides an
integer (a code, a block scale) the decision is taken in fp32, the precision
the CUDA kernels use, with the exact op sequence written out below.

Readings of the pages (where they are silent or garbled) are marked READING.

Parity status: every public function is pinned by a CPU test in
``tests/test_oracle_*.py`` (see each function's "Pinned by" line).
"""
from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# Formats  ([outlier §1.1] E2M1 spans [-6, 6]; [msr §一, §六] E2M1 = 2 exponent
# bits + 1 mantissa bit, 16 values; [lowprec §1.1] E4M3 and E8M0 scales)
# ----------------------------------------------------------------------------

#: magnitudes of the eight non-negative E2M1 codes 0..7
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

MXFP4 = 0
NVFP4 = 1
BLOCK = {MXFP4: 32, NVFP4: 16}

#: 6 * 448: largest E2M1 magnitude times largest finite E4M3 value
NVFP4_TENSOR_DIVISOR = np.float32(2688.0)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each 4-bit E2M1 code (bit 3 = sign).  Pinned by test_e2m1_grid."""
    codes = np.asarray(codes, dtype=np.uint8) & 0xF
    mag = E2M1_GRID[codes & 7]
    return np.where(codes & 8, -mag, mag)


def e2m1_encode_rtn(xs: np.ndarray) -> np.ndarray:
    """Round-to-nearest onto the E2M1 grid ([outlier §4.1]: forward uses RTN).

    READING: ties go to the even code (the one whose mantissa bit is 0);
    magnitudes above 6 saturate to 6 (the grid's end, [outlier §1.1]); the
    sign bit is kept even when the magnitude rounds to 0 (IEEE conversion).
    Definition used: the nearest of the eight grid magnitudes, by exhaustive
    comparison.  Pinned by hand-derived tie points (tests/golden), an
    independent IEEE-rounding formulation over all bf16 values, idempotence.
    """
    xs = np.asarray(xs, dtype=np.float32)
    # saturate first: every magnitude above 6 has 6 as its nearest grid point,
    # and clamping keeps the fp64 distances below distinct for huge inputs
    a = np.minimum(np.abs(xs.astype(np.float64)), 7.0).reshape(-1, 1)
    dist = np.abs(a - E2M1_GRID.reshape(1, -1))            # [n, 8]
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best                                     # one or two adjacent candidates
    even = (np.arange(8) % 2 == 0).reshape(1, -1)
    cand_even = cand & even
    mag = np.where(cand_even.any(axis=1), cand_even.argmax(axis=1), cand.argmax(axis=1))
    sign = np.signbit(xs).reshape(-1).astype(np.uint8)
    return ((sign << 3) | mag.astype(np.uint8)).reshape(xs.shape)


def e2m1_encode_sr(xs: np.ndarray, u16: np.ndarray) -> np.ndarray:
    """Stochastic rounding onto the E2M1 grid.

    [lowprec §3.2] gives SR as floor(x) + (rand < frac); here "floor" is the
    largest grid point at or below |x| and frac is the position between that
    point and the next one (the grid is not uniform).  READING: rand is a
    16-bit uniform integer u16 and the test is u16 < frac * 65536, taken in
    fp32 (exact: frac is an exact fp32 value and 65536 a power of two).
    Magnitudes at or above 6 saturate to 6.  Sign kept as in RTN.
    Pinned by unbiasedness over many draws and fixed points on the grid.
    """
    xs = np.asarray(xs, dtype=np.float32)
    u16 = np.asarray(u16, dtype=np.uint32)
    a = np.minimum(np.abs(xs), np.float32(6.0))
    grid32 = E2M1_GRID.astype(np.float32)
    lo_code = np.searchsorted(grid32, a, side="right") - 1  # largest grid point <= a
    lo_code = np.clip(lo_code, 0, 7)
    hi_code = np.minimum(lo_code + 1, 7)
    lo = grid32[lo_code]
    hi = grid32[hi_code]
    step = np.where(hi_code > lo_code, hi - lo, np.float32(1.0)).astype(np.float32)
    frac = ((a - lo) / step).astype(np.float32)               # exact
    up = u16.astype(np.float32) < frac * np.float32(65536.0)
    mag = np.where((lo_code < 7) & up, hi_code, lo_code).astype(np.uint8)
    sign = np.signbit(xs).astype(np.uint8)
    return (sign << 3) | mag


def _e4m3_table() -> np.ndarray:
    """All non-negative finite E4M3 ("fn": bias 7, no infinities) values by byte."""
    vals = np.full(128, np.nan)
    for b in range(127):                                     # 0x7F is NaN
        e, m = b >> 3, b & 7
        vals[b] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_table()


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """Value of a non-negative E4M3 byte.  Pinned by test_e4m3_against_torch."""
    return E4M3_VALUES[np.asarray(b, dtype=np.uint8) & 0x7F]


def e4m3_encode_rn_satfinite(t: np.ndarray) -> np.ndarray:
    """Nearest non-negative finite E4M3 value, ties to even, saturating at 448.

    The NVFP4 block-scale encoding ([lowprec §1.1] E4M3 = 4 exponent and 3
    mantissa bits).  Exhaustive nearest search over the 127 finite values.
    Pinned against torch's float8_e4m3fn cast on inputs <= 448.
    """
    shape = np.shape(t)
    # satfinite: everything above 448 maps to 448 (clamped before the search)
    t = np.minimum(np.asarray(t, dtype=np.float32).astype(np.float64), 449.0).reshape(-1, 1)
    table = E4M3_VALUES[:127].reshape(1, -1)
    dist = np.abs(t - table)
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    even = (np.arange(127) % 2 == 0).reshape(1, -1)
    cand_even = cand & even
    b = np.where(cand_even.any(axis=1), cand_even.argmax(axis=1), cand.argmax(axis=1))
    return b.astype(np.uint8).reshape(shape)


def e8m0_exponent(amax: np.ndarray) -> np.ndarray:
    """MXFP4 block scale exponent e with scale = 2**e.

    READING of the printed rule "scale = 2^(floor(log2 amax)) - 2": the
    exponent is floor(log2 amax) - 2 (E2M1's largest exponent is 2, so
    amax / 2**e lies in [4, 8)).  floor(log2) is taken exactly from the binary
    exponent; e is clamped to the E8M0 range [-127, 127]; amax == 0 gives -127.
    Pinned by golden values and the [4, 8) invariant.
    """
    amax = np.asarray(amax, dtype=np.float32).astype(np.float64)
    _, ex = np.frexp(amax)                 # amax = m * 2**ex, m in [0.5, 1)
    e = ex.astype(np.int64) - 1 - 2
    e = np.where(amax == 0.0, -127, e)
    return np.clip(e, -127, 127)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 round-to-nearest-even, returned as fp32.  Pinned vs torch."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


# ----------------------------------------------------------------------------
# Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel
# random numbers: as easy as 1, 2, 3", SC'11), written from the paper.
# READING: the pages' SR snippet draws torch.rand_like; a counter-based
# generator is used so that a (seed, offset) pair reproduces SR bit for bit.
# ----------------------------------------------------------------------------
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)
_M32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """Ten Philox rounds.  ctr: 4 uint32 arrays, key: 2 uint32 values/arrays.

    Returns 4 uint32 arrays.  Pinned against the curand host generator.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _M32 for c in ctr)
    k0, k1 = (np.asarray(k, dtype=np.uint64) & _M32 for k in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _PHILOX_W0) & _M32
            k1 = (k1 + _PHILOX_W1) & _M32
        p0 = _PHILOX_M0 * c0
        p1 = _PHILOX_M1 * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & _M32,
                          (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & _M32)
    return tuple(c.astype(np.uint32) for c in (c0, c1, c2, c3))


def sr_uniform16(seed: int, offset: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """16-bit uniform for the element at linear output index idx.

    READING (pages silent): key = (seed low 32, seed high 32); Philox call
    n = offset + idx // 8 with counter (n low 32, n high 32, 0, stream);
    element idx takes 16-bit lane idx % 8 of the 128-bit output (word
    (idx % 8) // 2, low half for even idx).
    """
    idx = np.asarray(idx, dtype=np.uint64)
    n = np.uint64(offset) + (idx >> np.uint64(3))
    zeros = np.zeros_like(n)
    words = philox4x32_10((n & _M32, n >> np.uint64(32), zeros, zeros + np.uint64(stream)),
                          (np.uint64(seed) & _M32, np.uint64(seed) >> np.uint64(32)))
    lane = (idx & np.uint64(7)).astype(np.int64)
    w = np.choose(lane >> 1, words)
    return ((w >> ((lane & 1) * 16).astype(np.uint32)) & 0xFFFF).astype(np.uint16)


# ----------------------------------------------------------------------------
# 16-point random Hadamard transform ([outlier §4.1]: backward operands get an
# RHT before SR quantization; 16 points and Rademacher signs are the plainest
# reading of "RHT" with 16-element NVFP4 blocks).
# ----------------------------------------------------------------------------

def rht16_signs(seed: int) -> np.ndarray:
    """sigma_j = -1 where bit j of Philox(key=seed, counter=0) word 0 is set."""
    w0 = int(philox4x32_10((0, 0, 0, 0), (seed & 0xFFFFFFFF, seed >> 32))[0])
    return np.array([-1.0 if (w0 >> j) & 1 else 1.0 for j in range(16)], dtype=np.float32)


def rht16_chunks(v: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """y = 1/4 * H16 * diag(signs) * v on the last axis (length 16), in fp32.

    The Walsh-Hadamard butterfly runs with strides 1, 2, 4, 8 in that order; the
    fp32 operation order is fixed by that loop.  Pinned against
    scipy.linalg.hadamard, orthogonality and norm preservation.
    """
    v = (np.asarray(v, dtype=np.float32) * signs.astype(np.float32)).astype(np.float32)
    v = v.copy()
    for h in (1, 2, 4, 8):
        for i in range(16):
            if i & h:
                continue
            a = v[..., i].copy()
            b = v[..., i + h].copy()
            v[..., i] = a + b
            v[..., i + h] = a - b
    return (v * np.float32(0.25)).astype(np.float32)


def rht16(x: np.ndarray, axis: int, seed: int) -> np.ndarray:
    """RHT16 applied to consecutive 16-element chunks along ``axis`` (0 or 1)."""
    x = np.asarray(x, dtype=np.float32)
    w = x if axis == 1 else x.T
    r, c = w.shape
    assert c % 16 == 0
    y = rht16_chunks(w.reshape(r, c // 16, 16), rht16_signs(seed)).reshape(r, c)
    return y if axis == 1 else np.ascontiguousarray(y.T)


# ----------------------------------------------------------------------------
# Quantizer  Q(x) = s * round(x / s)   ([grad §2.1])
# ----------------------------------------------------------------------------

def nvfp4_tensor_scale(amax_t) -> np.float32:
    """Per-tensor fp32 scale g = amax_t / (6 * 448), one fp32 division."""
    return np.float32(np.float32(amax_t) / NVFP4_TENSOR_DIVISOR)


def tensor_amax(x: np.ndarray) -> np.float32:
    return np.float32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) if x.size else np.float32(0)


def _block_amax(w: np.ndarray, bsz: int, two_d: bool) -> np.ndarray:
    """Block amax (fp32), one value per block: [R, C/bsz] for 1D blocks along
    the last axis, [R/16, C/16] for 16x16 tiles."""
    r, c = w.shape
    a = np.abs(w)
    if not two_d:
        return a.reshape(r, c // bsz, bsz).max(axis=2)
    return a.reshape(r // 16, 16, c // 16, 16).max(axis=(1, 3))


def _per_element(m: np.ndarray, bsz: int, two_d: bool) -> np.ndarray:
    """A per-block array spread over the block's elements (1D: bsz along the
    last axis; 2D: 16 x 16)."""
    if not two_d:
        return np.repeat(m, bsz, axis=1)
    return np.repeat(np.repeat(m, 16, axis=0), 16, axis=1)


def element_scale_inputs(fmt, amax_b, g):
    """Block scale byte and the fp32 multiplier applied to each element.

    MXFP4: byte = e + 127, multiplier 2**-e (exact).
    NVFP4 (READING, op for op in fp32):
        d = 6 * g ; t = amax_b / d ; sb = E4M3_rn_satfinite(t)
        s = dec(sb) * g ; r = 1 / s ; xs = x * r   (s == 0: codes are 0)
    Returns (scale_byte, multiplier r, s_is_zero mask).
    """
    if fmt == MXFP4:
        e = e8m0_exponent(amax_b)
        return (e + 127).astype(np.uint8), np.ldexp(1.0, -e).astype(np.float32), \
            np.zeros(np.shape(amax_b), dtype=bool)
    g = np.float32(g)
    if g == 0:
        z = np.zeros(np.shape(amax_b))
        return z.astype(np.uint8), z.astype(np.float32), np.ones(np.shape(amax_b), dtype=bool)
    d = np.float32(np.float32(6.0) * g)
    t = (np.asarray(amax_b, dtype=np.float32) / d).astype(np.float32)
    sb = e4m3_encode_rn_satfinite(t).reshape(np.shape(amax_b))
    s = (e4m3_decode(sb).astype(np.float32) * g).astype(np.float32)
    zero = s == 0
    with np.errstate(divide="ignore"):
        r = np.where(zero, np.float32(0), (np.float32(1.0) / np.where(zero, 1, s))).astype(np.float32)
    return sb, r, zero


def quantize(x, fmt, rounding="rtn", scaling="1d", transpose=False, rht=False,
             sr_seed=0, sr_offset=0, sr_stream=0, rht_seed=0, given_amax=None, block=None):
    """Block-scaled FP4 quantization of a 2-D tensor.

    x: fp32 array [R, C] (bf16 inputs are widened exactly).
    Blocks run along C, or along R when transpose=True; the output is then
    laid out [C, R] so that the blocked axis is contiguous.
    fmt MXFP4: 32-element blocks, E8M0 scale; NVFP4: 16-element blocks, E4M3
    scale times a per-tensor fp32 scale g ([lowprec §1.1]).
    rounding 'rtn' (forward) or 'sr' (backward) ([outlier §4.1]).
    block: elements per scale (default the format's 32 / 16; [grad §4.2]
    studies 16-128 for either scale format: block sizes are a parameter).
    scaling '1d' or '2d' (one scale per 16x16 tile, [outlier §4.1-4.2],
    NVFP4 only).  rht: RHT16 along the blocked axis first ([outlier §4.1]).

    Returns (codes uint8 [R', C'/2] with the even element in the low nibble,
             scales uint8 [R', C'/B] (2D scales repeated over the 16 rows),
             g float32 or None).
    """
    bsz = block or BLOCK[fmt]
    w = np.asarray(x, dtype=np.float32)
    if transpose:
        w = np.ascontiguousarray(w.T)
    r, c = w.shape
    assert c % bsz == 0
    two_d = scaling == "2d"
    if two_d:
        assert fmt == NVFP4 and r % 16 == 0
    if rht:
        w = rht16(w, axis=1, seed=rht_seed)
    g = None
    if fmt == NVFP4:
        amax_t = tensor_amax(w) if given_amax is None else np.float32(given_amax)
        g = nvfp4_tensor_scale(amax_t)
    amax_b = _block_amax(w, bsz, two_d)                     # per block
    sb_blk, mult_blk, zero_blk = element_scale_inputs(fmt, amax_b, g)
    mult = _per_element(mult_blk, bsz, two_d)
    zero = _per_element(zero_blk, bsz, two_d)
    xs = (w * mult).astype(np.float32)
    if rounding == "rtn":
        codes = e2m1_encode_rtn(xs)
    else:
        idx = np.arange(r * c, dtype=np.uint64).reshape(r, c)
        codes = e2m1_encode_sr(xs, sr_uniform16(sr_seed, sr_offset, sr_stream, idx))
    codes = np.where(zero, np.uint8(0), codes).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    # one byte per block; 2D tiles repeat theirs over the tile's 16 rows
    scales = (np.repeat(sb_blk, 16, axis=0) if two_d else sb_blk).astype(np.uint8)
    return packed, scales, g


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def block_scale_values(scales, fmt) -> np.ndarray:
    """Decoded block scales (fp64, exact), without the NVFP4 tensor scale."""
    scales = np.asarray(scales, dtype=np.uint8)
    if fmt == MXFP4:
        return np.ldexp(1.0, scales.astype(np.int64) - 127)
    return e4m3_decode(scales)


def dequantize(packed, scales, fmt, g=None, block=None) -> np.ndarray:
    """x_hat = code value * s  ([grad §2.1]), returned in fp32.

    MXFP4: cv * 2**e (exact).  NVFP4: fp32(fp32(cv * dec(sb)) * g); the inner
    product of a 2-bit and a 4-bit significand is exact, so one rounding.
    """
    bsz = block or BLOCK[fmt]
    cv = e2m1_decode(unpack_codes(packed))
    sv = np.repeat(block_scale_values(scales, fmt), bsz, axis=1)
    v = (cv * sv).astype(np.float32)
    if fmt == NVFP4:
        v = (v * np.float32(g)).astype(np.float32)
    return v


def operand_values(packed, scales, fmt) -> np.ndarray:
    """Exact fp64 values the MMA multiplies: code value * block scale (no g)."""
    bsz = BLOCK[fmt]
    return e2m1_decode(unpack_codes(packed)) * np.repeat(block_scale_values(scales, fmt), bsz, axis=1)


# ----------------------------------------------------------------------------
# Differentiable gradient estimator ([msr §二]): the quantizer is replaced in
# the backward pass by f(x) = d/2 (1 + sign(2x/d - 1) |2x/d - 1|^(1/k)) on each
# quantization interval of width d, whose derivative is clamped at 3.0.
# ----------------------------------------------------------------------------

def dge_derivative(xs: np.ndarray, k: float, clamp: float, outside: float = 1.0) -> np.ndarray:
    """f'(xs) on the E2M1 grid, fp64.

    Local coordinate u = 2(|xs| - g_i)/d - 1 on the interval [g_i, g_i + d)
    holding |xs|; f' = min(clamp, (1/k) |u|^(1/k - 1)) and u == 0 gives clamp.
    READING: |xs| >= 6 lies outside every interval and gets ``outside``
    (1.0 = straight-through estimator, [grad §3.1]).
    """
    a = np.abs(np.asarray(xs, dtype=np.float32).astype(np.float64))
    lo_code = np.clip(np.searchsorted(E2M1_GRID, a, side="right") - 1, 0, 6)
    lo = E2M1_GRID[lo_code]
    d = E2M1_GRID[lo_code + 1] - lo
    u = 2.0 * (a - lo) / d - 1.0
    au = np.abs(u)
    with np.errstate(divide="ignore"):
        raw = np.where(au == 0.0, np.inf, (1.0 / k) * np.power(np.where(au == 0, 1.0, au), 1.0 / k - 1.0))
    fp = np.minimum(clamp, raw)
    return np.where(a >= 6.0, outside, fp)


def scaled_inputs(x, scales, fmt, g=None, block=None) -> np.ndarray:
    """xs = x / s exactly as the quantizer forms it (fp32), from stored scales."""
    bsz = block or BLOCK[fmt]
    w = np.asarray(x, dtype=np.float32)
    sb = np.repeat(np.asarray(scales, dtype=np.uint8), bsz, axis=1)
    if fmt == MXFP4:
        return (w * np.ldexp(1.0, 127 - sb.astype(np.int64)).astype(np.float32)).astype(np.float32)
    s = (e4m3_decode(sb).astype(np.float32) * np.float32(g)).astype(np.float32)
    zero = s == 0
    r = np.where(zero, np.float32(0), np.float32(1.0) / np.where(zero, 1, s)).astype(np.float32)
    return (w * r).astype(np.float32)


def dge_backward(x, scales, fmt, g, dy, k=5.0, clamp=3.0, outside=1.0) -> np.ndarray:
    """dx = dy * f'(x / s) for x quantized along its rows; fp64 result."""
    xs = scaled_inputs(x, scales, fmt, g)
    return np.asarray(dy, dtype=np.float64) * dge_derivative(xs, k, clamp, outside)


# ----------------------------------------------------------------------------
# Sigmoid-smoothed quantizer ([grad §3.2]):
#   Q_soft(x) = sum_i v_i sigma(beta (x - c_i)),
#   dQ_soft/dx = beta sum_i v_i sigma(beta (x - c_i)) (1 - sigma(beta (x - c_i)))
# READING: the page calls v_i "the quantization levels" and c_i "the interval
# midpoints" and says Q_soft tends to the standard quantizer as beta grows.
# The reading under which that limit holds: over the 15 signed E2M1 levels
# q_0 < ... < q_14 (-6 .. 6), c_i = (q_i + q_{i+1}) / 2 are the 14 decision
# thresholds, v_i = q_{i+1} - q_i the level steps, and the sum starts from the
# lowest level q_0: Q_soft(x) = q_0 + sum_i v_i sigma(beta (x - c_i)).  Each
# sigmoid then switches one step on as x crosses c_i, so beta -> inf gives
# round-to-nearest onto the grid, saturating at +-6.  The derivative is the
# page's expression with these v_i, c_i (the constant q_0 drops out).  Like
# the DGE, the smoothing acts on the scaled value x / s and the block scale s
# is held constant: y = s Q_soft(x / s), dx = dy Q_soft'(x / s).
# ----------------------------------------------------------------------------

def soft_grid():
    """(levels q_0..q_14, thresholds c_0..c_13, steps v_0..v_13), fp64."""
    q = np.concatenate([-E2M1_GRID[:0:-1], E2M1_GRID])      # -6 .. -0.5, 0, 0.5 .. 6
    c = 0.5 * (q[:-1] + q[1:])
    v = q[1:] - q[:-1]
    return q, c, v


def _sigmoid(z: np.ndarray) -> np.ndarray:
    """1 / (1 + e^-z) in fp64; e^-z overflowing to inf gives the limit 0."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def soft_quantize_scaled(xs: np.ndarray, beta: float) -> np.ndarray:
    """Q_soft(xs) = q_0 + sum_i v_i sigma(beta (xs - c_i)), fp64.  Pinned by
    test_soft_* (RTN limit, finite differences, odd symmetry, beta -> 0)."""
    q, c, v = soft_grid()
    z = float(beta) * (np.asarray(xs, dtype=np.float64)[..., None] - c)
    return q[0] + (v * _sigmoid(z)).sum(axis=-1)


def soft_derivative(xs: np.ndarray, beta: float) -> np.ndarray:
    """beta sum_i v_i sigma(z_i) (1 - sigma(z_i)), z_i = beta (xs - c_i), fp64.
    1 - sigma(z) is evaluated as sigma(-z) (the same number) so that the tails
    keep their relative precision."""
    _, c, v = soft_grid()
    z = float(beta) * (np.asarray(xs, dtype=np.float64)[..., None] - c)
    return float(beta) * (v * _sigmoid(z) * _sigmoid(-z)).sum(axis=-1)


def block_scales_expanded(scales, fmt, g=None, block=None) -> np.ndarray:
    """The block scale s of every element (fp32 values as the quantizer formed
    them: 2^(e-127) for E8M0, e4m3(b) * g for NVFP4), expanded along the row."""
    bsz = block or BLOCK[fmt]
    sb = np.repeat(np.asarray(scales, dtype=np.uint8), bsz, axis=1)
    if fmt == MXFP4:
        return np.ldexp(1.0, sb.astype(np.int64) - 127).astype(np.float32)
    return (e4m3_decode(sb).astype(np.float32) * np.float32(g)).astype(np.float32)


def soft_forward(x, scales, fmt, g, beta, block=None) -> np.ndarray:
    """y = s Q_soft(x / s) for x quantized along its rows; fp64 result."""
    xs = scaled_inputs(x, scales, fmt, g, block)
    s = block_scales_expanded(scales, fmt, g, block).astype(np.float64)
    return s * soft_quantize_scaled(xs, beta)


def soft_backward(x, scales, fmt, g, dy, beta) -> np.ndarray:
    """dx = dy Q_soft'(x / s) for x quantized along its rows; fp64 result."""
    xs = scaled_inputs(x, scales, fmt, g)
    return np.asarray(dy, dtype=np.float64) * soft_derivative(xs, beta)


# ----------------------------------------------------------------------------
# Block-scaled GEMM  Y[M, N] = sum_k A[m, k] B[n, k]   (fp64 accumulation)
# ----------------------------------------------------------------------------

def gemm(a_codes, a_scales, b_codes, b_scales, fmt, g_a=None, g_b=None):
    """Returns (Y, bound) with bound = sum_k |A||B| for the error tolerance."""
    A = operand_values(a_codes, a_scales, fmt)
    B = operand_values(b_codes, b_scales, fmt)
    alpha = 1.0 if fmt == MXFP4 else float(np.float32(g_a)) * float(np.float32(g_b))
    return alpha * (A @ B.T), alpha * (np.abs(A) @ np.abs(B).T)


# ----------------------------------------------------------------------------
# Hot-channel compensation ([outlier §3.1-3.2, §4.1])
#   W^T X (quantized) = W^T X + (W^T dX + dW^T X) + dW^T dX  (error split)
# READING: "S-O2-B" = single GEMM, second order, BF16 residual columns.  With
# dX = X - X_hat and dW = W - W_hat, the extra K columns
#   A_ext = [dX_H | X_H],  B_ext = [W_hat_H | dW_H]
# make Y = X_hat W_hat^T + A_ext B_ext^T equal, on the hot channels H, to the
# unquantized product.  Order 1 is the page's literal concat:
#   A_ext = [X_H], B_ext = [dW_H].
# B_ext is pre-divided by alpha = g_X g_W so that one accumulator holds both
# parts and the epilogue multiplies everything by alpha.
# ----------------------------------------------------------------------------

def hcp_channel_errors(x, x_codes, x_scales, fmt, g=None) -> np.ndarray:
    """e_c = sum_m (X[m, c] - X_hat[m, c])^2 in fp64 ("largest quantization error")."""
    xh = dequantize(x_codes, x_scales, fmt, g).astype(np.float64)
    return ((np.asarray(x, dtype=np.float64) - xh) ** 2).sum(axis=0)


def hcp_top_channels(e, k_hot: int) -> np.ndarray:
    """The k_hot channels with the largest error e_c, ties to the lower index,
    in ascending order ([outlier §4.1]: top 9% of channels)."""
    e = np.asarray(e, dtype=np.float64)
    order = sorted(range(len(e)), key=lambda c: (-e[c], c))
    return np.array(sorted(order[:k_hot]), dtype=np.int32)


def hcp_select(x, x_codes, x_scales, fmt, g, k_hot: int) -> np.ndarray:
    """Indices of the k_hot channels with the largest quantization error."""
    return hcp_top_channels(hcp_channel_errors(x, x_codes, x_scales, fmt, g), k_hot)


def hcp_num_hot(k: int, ratio: float = 0.09) -> int:
    """h = ceil(ratio * K)  (READING of "top 9%")."""
    return int(math.ceil(ratio * k))


def hcp_extra_operands(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order=2):
    """bf16-valued extra K columns (returned as fp32 arrays of bf16 values)."""
    hot = np.asarray(hot, dtype=np.int64)
    xf = np.asarray(x, dtype=np.float32)[:, hot]
    wf = np.asarray(w, dtype=np.float32)[:, hot]
    xh = dequantize(x_codes, x_scales, fmt, g_x)[:, hot]
    wh = dequantize(w_codes, w_scales, fmt, g_w)[:, hot]
    if fmt == NVFP4:
        alpha = np.float32(np.float32(g_x) * np.float32(g_w))
        inv_alpha = np.float32(np.float32(1.0) / alpha)
    else:
        inv_alpha = np.float32(1.0)
    dx = (xf - xh).astype(np.float32)
    dw = (wf - wh).astype(np.float32)
    if order == 2:
        a_ext = np.concatenate([bf16_round(dx), bf16_round(xf)], axis=1)
        b_ext = np.concatenate([bf16_round((wh * inv_alpha).astype(np.float32)),
                                bf16_round((dw * inv_alpha).astype(np.float32))], axis=1)
    elif order == 1:
        a_ext = bf16_round(xf)
        b_ext = bf16_round((dw * inv_alpha).astype(np.float32))
    else:
        raise ValueError("order must be 1 or 2")
    return a_ext.astype(np.float32), b_ext.astype(np.float32)


def hcp_gemm(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order=2):
    """Y = alpha (X_hat W_hat^T + A_ext B_ext^T) in fp64; returns (Y, bound)."""
    A = operand_values(x_codes, x_scales, fmt)
    B = operand_values(w_codes, w_scales, fmt)
    a_ext, b_ext = hcp_extra_operands(x, x_codes, x_scales, w, w_codes, w_scales,
                                      fmt, g_x, g_w, hot, order)
    # the FP4 part carries g_x g_w exactly; the residual part was divided by the
    # fp32 product alpha, so it is multiplied back by that same fp32 value
    alpha = 1.0 if fmt == MXFP4 else float(np.float32(g_x)) * float(np.float32(g_w))
    alpha32 = 1.0 if fmt == MXFP4 else float(np.float32(np.float32(g_x) * np.float32(g_w)))
    ae = a_ext.astype(np.float64)
    be = b_ext.astype(np.float64)
    y = alpha * (A @ B.T) + alpha32 * (ae @ be.T)
    bound = alpha * (np.abs(A) @ np.abs(B).T) + alpha32 * (np.abs(ae) @ np.abs(be).T)
    return y, bound


def gemm_tolerance(bound, y_ref, out_bf16: bool):
    """|Y - Y_ref| <= 1e-3 * sum|a||b|, plus 2^-8 |Y_ref| for a bf16 output.

    READING: the pages fix no output precision; bf16 keeps an 8-bit
    significand, so rounding the result to bf16 moves it by up to 2^-8 of its
    magnitude on top of the accumulation bound.
    """
    tol = 1e-3 * np.asarray(bound)
    if out_bf16:
        tol = tol + 2.0 ** -8 * np.abs(y_ref)
    return tol


# ----------------------------------------------------------------------------
# Outlier clamping and compensation, OCC ([msr §三, §六])
#   The largest 1% of activation magnitudes are outliers: the 99% quantile of
#   |X| is the threshold tau, X is clamped to [-tau, tau] before it is
#   quantized, and the clamped-away part dX = X - clamp(X) (a sparse matrix)
#   goes through a high-precision product beside the FP4 GEMM:
#       Y = Q(X_c) Q(W)^T + dX W^T.
# READING: the quantile is taken over the magnitudes of the whole tensor, by
# nearest rank (tau = the ceil(q n)-th smallest |x|, so that at least q n
# magnitudes are <= tau); elements with |x| > tau are the outliers.  W in the
# compensation is the unquantized weight (bf16 values), the high-precision
# operand; the quality numbers (cosine, MSE, SNR) compare X with its
# reconstruction dequant(Q(X_c)) + dX (OCC) or dequant(Q(X)) (direct).
# ----------------------------------------------------------------------------

def occ_threshold(x, q: float = 0.99) -> np.float32:
    """tau: the ceil(q n)-th smallest |x| (1-based rank) over all n elements."""
    a = np.sort(np.abs(np.asarray(x, dtype=np.float32)).reshape(-1), kind="stable")
    n = a.size
    rank = max(1, int(math.ceil(q * n)))
    return np.float32(a[rank - 1])


def occ_split(x, tau):
    """(X_c, dX) with X_c = min(max(x, -tau), tau) and dX = x - X_c, both fp32
    (dX is exact: x and tau are values of the input's own precision)."""
    w = np.asarray(x, dtype=np.float32)
    t = np.float32(tau)
    xc = np.minimum(np.maximum(w, -t), t).astype(np.float32)
    return xc, (w - xc).astype(np.float32)


def occ_outliers(x, tau):
    """Outlier positions (row, col), row-major order, and their dX values."""
    _, dx = occ_split(x, tau)
    rows, cols = np.nonzero(np.abs(np.asarray(x, dtype=np.float32)) > np.float32(tau))
    return rows, cols, dx[rows, cols]


def occ_gemm(x, w, fmt, tau):
    """Y = alpha Q(X_c) Q(W)^T + dX W^T in fp64 (W: its bf16/fp32 values).

    Returns (Y, bound, (xc_codes, xc_scales, g_x), (w_codes, w_scales, g_w))
    with bound = sum_k |a||b| of the FP4 part plus sum_k |dX||W|."""
    xc, dx = occ_split(x, tau)
    xq = quantize(xc, fmt)
    wq = quantize(w, fmt)
    y, bound = gemm(xq[0], xq[1], wq[0], wq[1], fmt, xq[2], wq[2])
    wf = np.asarray(w, dtype=np.float64)
    dxf = dx.astype(np.float64)
    return y + dxf @ wf.T, bound + np.abs(dxf) @ np.abs(wf).T, xq, wq


def quant_error_stats(x, x_hat):
    """Cosine similarity, mean squared error and SNR (dB) of x_hat against x,
    fp64: cos = <x, x_hat> / (|x| |x_hat|), MSE = mean (x - x_hat)^2,
    SNR = 10 log10(sum x^2 / sum (x - x_hat)^2)."""
    a = np.asarray(x, dtype=np.float64).reshape(-1)
    b = np.asarray(x_hat, dtype=np.float64).reshape(-1)
    err = ((a - b) ** 2).sum()
    cos = float(a @ b / math.sqrt((a @ a) * (b @ b)))
    return {"cos": cos, "mse": float(err / a.size), "snr_db": float(10.0 * math.log10((a @ a) / err))}


def occ_reconstruction(x, fmt, tau):
    """dequant(Q(X_c)) + dX, fp64: what the OCC forward stands for."""
    xc, dx = occ_split(x, tau)
    codes, scales, g = quantize(xc, fmt)
    return dequantize(codes, scales, fmt, g).astype(np.float64) + dx.astype(np.float64)


def relative_error(x, x_hat) -> float:
    """||x - x_hat||_2 / ||x||_2 (fp64).  READING of the "relative error %"
    table of [grad §5.1]: the relative L2 error of the reconstruction."""
    a = np.asarray(x, dtype=np.float64).reshape(-1)
    b = np.asarray(x_hat, dtype=np.float64).reshape(-1)
    return float(np.sqrt(((a - b) ** 2).sum() / (a @ a)))


# ----------------------------------------------------------------------------
# Hot channels zeroed before quantizing: a variant of hot-channel compensation
# ([outlier §3.1-3.2]).  READING: the hot channels H leave the FP4 operand
# altogether -- X_H is set to 0 before X is quantized, so the hot channels no
# longer inflate the scales of the blocks they sit in -- and their whole
# product goes through the bf16 extra K columns:
#     Y = alpha Q(X_0) Q(W)^T + X_H W_H^T,   X_0 = X with the columns H zeroed.
# As in the compensated GEMM, B_ext is pre-divided by alpha so that one fp32
# scaling of the accumulator serves both parts: A_ext = bf16(X_H),
# B_ext = bf16(W_H / alpha).  NVFP4's tensor scale is that of X_0.
# ----------------------------------------------------------------------------

def hcp_zero_columns(x, hot) -> np.ndarray:
    """X_0: x with the columns in `hot` set to 0 (fp32)."""
    x0 = np.array(x, dtype=np.float32, copy=True)
    x0[:, np.asarray(hot, dtype=np.int64)] = 0.0
    return x0


def hcp_zeroed_operands(x, w, fmt, g_x, g_w, hot):
    """(A_ext, B_ext) = (bf16(X_H), bf16(W_H / alpha)) as fp32 arrays of bf16 values."""
    hot = np.asarray(hot, dtype=np.int64)
    if fmt == NVFP4:
        inv_alpha = np.float32(np.float32(1.0) / np.float32(np.float32(g_x) * np.float32(g_w)))
    else:
        inv_alpha = np.float32(1.0)
    a_ext = bf16_round(np.asarray(x, dtype=np.float32)[:, hot])
    b_ext = bf16_round((np.asarray(w, dtype=np.float32)[:, hot] * inv_alpha).astype(np.float32))
    return a_ext.astype(np.float32), b_ext.astype(np.float32)


def hcp_zeroed_gemm(x, w, fmt, hot):
    """Y = alpha Q(X_0) Q(W)^T + A_ext B_ext^T alpha32 in fp64; returns
    (Y, bound, (x0 codes, scales, g), (w codes, scales, g))."""
    x0q = quantize(hcp_zero_columns(x, hot), fmt)
    wq = quantize(w, fmt)
    y, bound = gemm(x0q[0], x0q[1], wq[0], wq[1], fmt, x0q[2], wq[2])
    a_ext, b_ext = hcp_zeroed_operands(x, w, fmt, x0q[2], wq[2], hot)
    alpha32 = 1.0 if fmt == MXFP4 else float(np.float32(np.float32(x0q[2]) * np.float32(wq[2])))
    ae, be = a_ext.astype(np.float64), b_ext.astype(np.float64)
    return y + alpha32 * (ae @ be.T), bound + alpha32 * (np.abs(ae) @ np.abs(be).T), x0q, wq


# ----------------------------------------------------------------------------
# FP8 (E4M3) residual columns for the compensated GEMM ([outlier §3.1]'s extra
# K columns; the MSR write-up §六 runs its high-precision sparse compensation
# in FP8).  READING: every row of A_ext and of B_ext gets its own fp32 scale
# s = amax(row) / 448 and each value becomes the nearest E4M3 value of v / s
# (ties to even, saturating at 448, sign kept); the residual product
# sum_j A_ext[m, j] B_ext[n, j] is then s_A[m] s_B[n] sum_j a8[m, j] b8[n, j],
# added by a second GEMM (C += ...).  The columns are those of the bf16 tail
# without the division by alpha (the row scales carry the magnitudes):
#   order 2: A = [dX_H | X_H], B = [W_hat_H | dW_H];  order 1: A = X_H, B = dW_H;
#   order 0 (hot channels zeroed in X): A = X_H, B = W_H.
# ----------------------------------------------------------------------------

def e4m3_rows(v):
    """(values, scales): per-row E4M3 rounding of v [R, C] with s = fp32(amax / 448);
    values are the decoded E4M3 numbers (fp64, without s).  All-zero rows: s = 0."""
    v = np.asarray(v, dtype=np.float32)
    amax = np.abs(v).max(axis=1) if v.shape[1] else np.zeros(v.shape[0], np.float32)
    s = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    t = (np.abs(v) / safe[:, None]).astype(np.float32)
    mag = e4m3_decode(e4m3_encode_rn_satfinite(t))
    vals = np.where(np.signbit(v), -mag, mag)
    vals = np.where(s[:, None] == 0, 0.0, vals)
    return vals.astype(np.float64), s


def hcp_fp8_columns(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order=2):
    """fp32 values of the extra columns (before the E4M3 rounding), per order."""
    hot = np.asarray(hot, dtype=np.int64)
    xf = np.asarray(x, dtype=np.float32)[:, hot]
    wf = np.asarray(w, dtype=np.float32)[:, hot]
    xh = dequantize(x_codes, x_scales, fmt, g_x)[:, hot]
    wh = dequantize(w_codes, w_scales, fmt, g_w)[:, hot]
    dx = (xf - xh).astype(np.float32)
    dw = (wf - wh).astype(np.float32)
    if order == 2:
        return np.concatenate([dx, xf], axis=1), np.concatenate([wh, dw], axis=1)
    if order == 1:
        return xf, dw
    if order == 0:
        return xf, wf
    raise ValueError("order must be 0, 1 or 2")


def hcp_gemm_fp8(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order=2):
    """Y = alpha Q(X) Q(W)^T + s_A s_B (a8 b8^T) in fp64; returns (Y, bound).
    For order 0, x_codes / x_scales / g_x are the quantization of X with H zeroed."""
    y, bound = gemm(x_codes, x_scales, w_codes, w_scales, fmt, g_x, g_w)
    a, b = hcp_fp8_columns(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order)
    a8, sa = e4m3_rows(a)
    b8, sb = e4m3_rows(b)
    A = a8 * sa.astype(np.float64)[:, None]
    B = b8 * sb.astype(np.float64)[:, None]
    return y + A @ B.T, bound + np.abs(A) @ np.abs(B).T


# ----------------------------------------------------------------------------
# HCP extra columns as MXFP8 in the FP4 accumulator (single kernel)
#
# READING (the pages fix no FP8 format for the compensation: [msr] §六 runs its
# compensation in FP8, [lowprec] §1.1 describes the MX family, elements sharing
# a power-of-two E8M0 scale per 32): the extra columns of the bf16 tail, with
# B already divided by alpha but not rounded to bf16, are quantized along the
# hot-channel axis in blocks of 32.  Each part of the columns (order 2: [dX_H |
# X_H] and [W_hat_H | dW_H]) is padded with zeros to a multiple of 32 so that
# no block mixes the two parts.  A block's scale is 2^e with e the smallest
# integer such that amax / 2^e <= 448 (E4M3's largest value, so no element
# saturates), clamped to E8M0's [-127, 127] (amax 0: -127); each element is
# the nearest E4M3 value of v / 2^e, ties to even, sign kept.  A block-scaled
# FP8 MMA multiplies the columns into the FP4 part's accumulator:
#   Y = alpha (X_hat W_hat^T + sum_j a8[m,j] 2^ea[m,j/32] b8[n,j] 2^eb[n,j/32]).
# ----------------------------------------------------------------------------

def mxfp8_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest e with amax / 2**e <= 448, clamped to [-127, 127]; amax 0 -> -127.

    amax = m * 2**x with m in [0.5, 1) (frexp, exact): amax / 2**(x - 9) = 512 m
    lies in [256, 512), at most 448 exactly when m <= 7/8.  Pinned by a brute-force
    search over exponents and hand-derived points."""
    amax = np.asarray(amax, dtype=np.float32).astype(np.float64)
    m, x = np.frexp(amax)
    e = x.astype(np.int64) - 9 + (m > 0.875).astype(np.int64)
    e = np.where(amax == 0.0, -127, e)
    return np.clip(e, -127, 127)


def mxfp8_quantize_rows(v, block: int = 32):
    """v [R, C] (C a multiple of `block`) -> (codes uint8 [R, C], exps int [R, C / block]):
    E4M3 bytes (bit 7 the sign) of v / 2**e and the blocks' exponents e."""
    v = np.asarray(v, dtype=np.float32)
    R, C = v.shape
    blocks = v.reshape(R, C // block, block)
    amax = np.abs(blocks).max(axis=2) if C else np.zeros((R, 0), np.float32)
    e = mxfp8_exponent(amax)
    # v * 2**-e: the exact product rounded once to fp32
    t = (np.abs(blocks).astype(np.float64) * np.exp2(-e.astype(np.float64))[:, :, None]).astype(np.float32)
    mag = e4m3_encode_rn_satfinite(t)
    sign = np.signbit(blocks).astype(np.uint8) << 7
    return (mag | sign).reshape(R, C).astype(np.uint8), e


def mxfp8_values(codes, exps, block: int = 32) -> np.ndarray:
    """fp64 values dec(code) * 2**e of mxfp8_quantize_rows' output."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = e4m3_decode(codes & 0x7F)
    val = np.where(codes & 0x80, -mag, mag)
    return val * np.repeat(np.exp2(np.asarray(exps, dtype=np.float64)), block, axis=1)


def hcp_mxfp8_columns(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order=2):
    """fp32 extra columns before the MXFP8 rounding, each part padded to a
    multiple of 32 with zeros: A [M, parts * kp], B [N, parts * kp] (B / alpha)."""
    a, b = hcp_fp8_columns(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order)
    if fmt == NVFP4:
        inv_alpha = np.float32(np.float32(1.0) / np.float32(np.float32(g_x) * np.float32(g_w)))
        b = (b * inv_alpha).astype(np.float32)
    k = len(np.asarray(hot))
    parts = 2 if order == 2 else 1
    kp = -(-k // 32) * 32

    def pad(v):
        out = np.zeros((v.shape[0], parts * kp), np.float32)
        for p in range(parts):
            out[:, p * kp: p * kp + k] = v[:, p * k: (p + 1) * k]
        return out
    return pad(a), pad(b)


def hcp_gemm_mxfp8(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order=2):
    """Y = alpha (Q(X) Q(W)^T + A8 B8^T) in fp64 (A8, B8 the MXFP8 columns'
    values); returns (Y, bound).  For order 0, x_codes / x_scales / g_x are the
    quantization of X with H zeroed."""
    A = operand_values(x_codes, x_scales, fmt)
    B = operand_values(w_codes, w_scales, fmt)
    a, b = hcp_mxfp8_columns(x, x_codes, x_scales, w, w_codes, w_scales, fmt, g_x, g_w, hot, order)
    A8 = mxfp8_values(*mxfp8_quantize_rows(a))
    B8 = mxfp8_values(*mxfp8_quantize_rows(b))
    alpha = 1.0 if fmt == MXFP4 else float(np.float32(g_x)) * float(np.float32(g_w))
    alpha32 = 1.0 if fmt == MXFP4 else float(np.float32(np.float32(g_x) * np.float32(g_w)))
    y = alpha * (A @ B.T) + alpha32 * (A8 @ B8.T)
    bound = alpha * (np.abs(A) @ np.abs(B).T) + alpha32 * (np.abs(A8) @ np.abs(B8).T)
    return y, bound
