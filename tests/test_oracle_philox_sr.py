"""Pins for the oracle's Philox generator and stochastic rounding (CPU only)."""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest

import oracle as o
from conftest import golden


def test_philox_known_answer_vectors():
    for row in golden("philox4x32_10_kat.txt"):
        v = [int(t, 16) for t in row]
        got = [int(w) for w in o.philox4x32_10(tuple(v[0:4]), tuple(v[4:6]))]
        assert got == v[6:10]


def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if path and os.path.exists(path):
            return ctypes.CDLL(path)
    return None


@pytest.mark.parametrize("seed", [0, 12345, (7 << 32) | 99])
def test_philox_matches_curand_host_generator(seed):
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not found")
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        n = 1 << 19                      # 2^17 blocks: counter word 0 takes values 0 and 1
        buf = (ctypes.c_uint32 * n)()
        assert lib.curandGenerate(gen, buf, ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    got = np.frombuffer(buf, dtype=np.uint32).reshape(-1, 4)
    # the host generator runs 65536 subsequences: block b has counter (b / 65536, 0, b % 65536, 0)
    b = np.arange(got.shape[0], dtype=np.uint64)
    sub = np.uint64(65536)
    mine = np.stack(o.philox4x32_10((b // sub, b * 0, b % sub, b * 0),
                                    (seed & 0xFFFFFFFF, seed >> 32)), axis=1)
    assert np.array_equal(mine, got)


def test_sr_uniform16_lane_mapping():
    seed, off, stream = 0x1234_5678_9ABC, 77, 3
    idx = np.arange(64, dtype=np.uint64)
    u = o.sr_uniform16(seed, off, stream, idx)
    for call in range(8):
        n = off + call
        w = [int(x) for x in o.philox4x32_10((n & 0xFFFFFFFF, n >> 32, 0, stream),
                                             (seed & 0xFFFFFFFF, seed >> 32))]
        halves = [h for word in w for h in (word & 0xFFFF, word >> 16)]
        assert list(u[8 * call: 8 * call + 8]) == halves


def test_sr_decision_is_exact_fraction():
    # Over all 65536 values of the 16-bit uniform, the number that round up is
    # ceil(frac * 65536): the SR rule floor + (rand < frac) of the low-precision
    # page §3.2 with a 2^-16-resolution rand.
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.uniform(-6, 6, 200), [0.3, 2.25, 4.5, 5.999, 1e-6]]).astype(np.float32)
    u = np.arange(65536, dtype=np.uint32)
    grid = o.E2M1_GRID
    for x in xs:
        codes = o.e2m1_encode_sr(np.full(65536, x, dtype=np.float32), u)
        vals = o.e2m1_decode(codes)
        a = abs(float(x))
        i = np.searchsorted(grid, a, side="right") - 1
        lo, hi = grid[i], grid[min(i + 1, 7)]
        frac = (a - lo) / (hi - lo)
        n_up = int(np.count_nonzero(np.abs(vals) == hi)) if hi != lo else 0
        assert n_up == int(np.ceil(frac * 65536))
        assert set(np.abs(vals)) <= {lo, hi}
        assert np.all(np.signbit(vals) == np.signbit(x)) or a == 0


def test_sr_unbiased_over_seeds():
    # E[Q(x)] = x (4 sigma + the 2^-16 resolution bias) over 10^4 draws
    rng = np.random.default_rng(2)
    xs = rng.uniform(-5.9, 5.9, 32).astype(np.float32)
    n = 10000
    idx = np.arange(n * 32, dtype=np.uint64)
    u = o.sr_uniform16(2024, 0, 0, idx).reshape(n, 32)
    vals = o.e2m1_decode(o.e2m1_encode_sr(np.broadcast_to(xs, (n, 32)), u))
    mean = vals.mean(axis=0)
    grid = o.E2M1_GRID
    for j, x in enumerate(xs):
        a = abs(float(x))
        i = np.searchsorted(grid, a, side="right") - 1
        d = grid[i + 1] - grid[i]
        p = (a - grid[i]) / d
        sigma = d * np.sqrt(p * (1 - p) / n)
        assert abs(mean[j] - x) <= 4 * sigma + d * 2.0 ** -16 + 1e-12


def test_sr_fixed_points_and_saturation():
    vals = o.e2m1_decode(np.arange(16)).astype(np.float32)
    u = np.full(16, 0, dtype=np.uint32)
    assert np.array_equal(o.e2m1_encode_sr(vals, u), np.arange(16, dtype=np.uint8))
    assert np.array_equal(o.e2m1_encode_sr(vals, u + 65535), np.arange(16, dtype=np.uint8))
    big = np.float32([7.0, -100.0])
    assert list(o.e2m1_encode_sr(big, np.array([0, 0]))) == [7, 15]


def test_sr_quantize_reproducible_and_offset_advances():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((32, 64)).astype(np.float32)
    a = o.quantize(x, o.NVFP4, rounding="sr", sr_seed=1, sr_offset=0)
    b = o.quantize(x, o.NVFP4, rounding="sr", sr_seed=1, sr_offset=0)
    c = o.quantize(x, o.NVFP4, rounding="sr", sr_seed=1, sr_offset=256)
    assert np.array_equal(a[0], b[0]) and not np.array_equal(a[0], c[0])
    assert np.array_equal(a[1], c[1])          # scales do not depend on the draw
