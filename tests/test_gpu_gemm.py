"""GPU <-> oracle parity for the tcgen05 block-scaled GEMM, through the C ABI.

Bound (per element): |Y - Y_ref| <= 1e-3 * sum_k |a||b|  (+ 2^-8 |Y_ref| for a
bf16 output: an 8-bit significand), Y_ref the fp64 sum of the dequantized operands.
The structured cases isolate the data path (all block scales 1), the A-side
scales, the B-side scales and the scale index along K.
"""
import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o

pytestmark = pytest.mark.gpu

FMT = {fp4.FP4_FMT_MXFP4: o.MXFP4, fp4.FP4_FMT_NVFP4: o.NVFP4}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    from fp4_block_scaled_e8m0_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    fp4.load_library()


def _run(a_np, b_np, fmt, out_dtype=torch.float32, ldc_pad=0, accumulate=None):
    a = torch.from_numpy(a_np).to(torch.bfloat16)
    b = torch.from_numpy(b_np).to(torch.bfloat16)
    qa = fp4.fp4_quantize(a.cuda(), fp4.quant_params(fmt))
    qb = fp4.fp4_quantize(b.cuda(), fp4.quant_params(fmt))
    M, N = a.shape[0], b.shape[0]
    ldc = N + ldc_pad
    out = torch.zeros((M, ldc), dtype=out_dtype, device="cuda")
    if accumulate is not None:
        out[:, :N] = torch.from_numpy(accumulate).to(out_dtype)
    fp4.fp4_gemm(qa, qb, out=out[:, :N] if ldc_pad else out, accumulate=accumulate is not None)
    torch.cuda.synchronize()
    got = out[:, :N].float().cpu().numpy().astype(np.float64)
    ca, sa, ga = o.quantize(a.float().numpy(), FMT[fmt])
    cb, sb, gb = o.quantize(b.float().numpy(), FMT[fmt])
    y, bound = o.gemm(ca, sa, cb, sb, FMT[fmt], ga, gb)
    if accumulate is not None:
        acc = torch.from_numpy(accumulate).to(out_dtype).float().numpy().astype(np.float64)
        y = y + acc
        bound = bound + np.abs(acc) * 2.0 ** -20
    return got, y, bound


def _assert_close(got, y, bound, out_dtype, label):
    tol = o.gemm_tolerance(bound, y, out_dtype == torch.bfloat16) + 1e-30
    err = np.abs(got - y)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)
        rows = np.unique(idx[:, 0])
        cols = np.unique(idx[:, 1])
        msg = [f"{label}: {bad.sum()} of {bad.size} outside the bound; rows {rows[:10]}..({len(rows)}), "
               f"cols {cols[:10]}..({len(cols)})"]
        for r, c in idx[:6]:
            msg.append(f"  [{r},{c}] got {got[r, c]:.6g} want {y[r, c]:.6g} tol {tol[r, c]:.3g}")
        raise AssertionError("\n".join(msg))


def _grid_matrix(rng, rows, k, bsz, row_exp=None, k_exp=None):
    """Values on the E2M1 grid times per-block powers of two, each block holding a
    6 so that its MXFP4 scale is exactly the chosen power of two."""
    codes = rng.integers(0, 16, (rows, k))
    v = o.e2m1_decode(codes)
    v[:, ::bsz] = 6.0
    e = np.zeros((rows, k // bsz))
    if row_exp is not None:
        e += row_exp.reshape(-1, 1)
    if k_exp is not None:
        e += k_exp.reshape(1, -1)
    return (v * np.repeat(2.0 ** e, bsz, axis=1)).astype(np.float32)


@pytest.mark.parametrize("case", ["unit", "a_rows", "b_rows", "k_blocks", "all"])
def test_gemm_structured_mxfp4(case):
    rng = np.random.default_rng(5)
    M, N, K = 128, 256, 256
    ra = rng.integers(-4, 5, M) if case in ("a_rows", "all") else None
    rb = rng.integers(-4, 5, N) if case in ("b_rows", "all") else None
    ka = rng.integers(-3, 4, K // 32) if case in ("k_blocks", "all") else None
    kb = rng.integers(-3, 4, K // 32) if case in ("k_blocks", "all") else None
    a = _grid_matrix(rng, M, K, 32, ra, ka)
    b = _grid_matrix(rng, N, K, 32, rb, kb)
    got, y, bound = _run(a, b, fp4.FP4_FMT_MXFP4)
    _assert_close(got, y, bound, torch.float32, f"mxfp4 structured {case}")


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("shape", [(128, 256, 64), (128, 256, 512), (256, 512, 512), (200, 300, 320),
                                   (64, 40, 96), (384, 640, 1024), (130, 520, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_matches_oracle(fmt, shape, out_dtype):
    M, N, K = shape
    if K % fp4.BLOCK[fmt]:
        pytest.skip("K not a multiple of the block")
    rng = np.random.default_rng(M * 7 + N * 3 + K + fmt)
    a = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-2, 2, (M, 1)))).astype(np.float32)
    b = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    pad = (-N) % 8
    got, y, bound = _run(a, b, fmt, out_dtype, ldc_pad=pad)
    _assert_close(got, y, bound, out_dtype, f"fmt={fmt} {shape} {out_dtype}")


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
@pytest.mark.parametrize("M,N,K", [(4000, 7400, 64), (4000, 7400, 256), (3130, 4296, 768)])
def test_gemm_many_tiles_per_cta(fmt, M, N, K):
    """The persistent tile loop: 928 (or 425) tiles, ragged in M and N, on at
    most one CTA per SM, with 1-3 K steps per tile, so each CTA's slab and
    scale rings wrap across tile boundaries; every element against the oracle,
    bf16 and fp32 out."""
    rng = np.random.default_rng(K + fmt)
    a = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-2, 2, (M, 1)))).astype(np.float32)
    b = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    at, bt = torch.from_numpy(a).to(torch.bfloat16), torch.from_numpy(b).to(torch.bfloat16)
    qa = fp4.fp4_quantize(at.cuda(), fp4.quant_params(fmt))
    qb = fp4.fp4_quantize(bt.cuda(), fp4.quant_params(fmt))
    ca, sa, ga = o.quantize(at.float().numpy(), FMT[fmt])
    cb, sb, gb = o.quantize(bt.float().numpy(), FMT[fmt])
    y, bound = o.gemm(ca, sa, cb, sb, FMT[fmt], ga, gb)
    for out_dtype in (torch.bfloat16, torch.float32):
        out = fp4.fp4_gemm(qa, qb, out=torch.empty((M, N), dtype=out_dtype, device="cuda"))
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        _assert_close(got, y, bound, out_dtype, f"fmt={fmt} {M}x{N}x{K} {out_dtype}")


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_MXFP4, fp4.FP4_FMT_NVFP4])
def test_gemm_accumulate(fmt):
    rng = np.random.default_rng(9)
    M, N, K = 256, 256, 512
    a = rng.standard_normal((M, K)).astype(np.float32)
    b = rng.standard_normal((N, K)).astype(np.float32)
    c0 = rng.standard_normal((M, N)).astype(np.float32)
    got, y, bound = _run(a, b, fmt, torch.float32, accumulate=c0)
    _assert_close(got, y, bound, torch.float32, "accumulate")


def test_gemm_status_clean_after_runs():
    assert fp4.fp4_sync_status() == fp4.FP4_OK
