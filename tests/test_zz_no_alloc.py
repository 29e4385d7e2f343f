"""fp4_hcp_select_noalloc: hot-channel selection that allocates nothing.

Some callers cannot allocate device memory -- their GPU memory belongs to their
own caching pool, or they cannot take the device-wide synchronization that
cudaMalloc/cudaFree may cause.  This entry point keeps its scratch in a fixed
array inside the library instead of a caller workspace.  The test calls it
through the C ABI several times in a row, on different tensors (so scratch left
over from one call would show in the next) and once on a side stream, with
both scale layouts, and compares each result with the workspace entry point
fp4_hcp_select under the selection tolerance the other tests use: the two sets
may differ only on channels whose error lies within 1e-5 (relative) of the
k-th largest, where fp32 sums taken in a different order can swap the ranking.
The edge cases (no rows, no hot channels) must give what fp4_hcp_select gives.
Collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp4_block_scaled_e8m0_gb300 as fp4
import oracle as o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import os
    from fp4_block_scaled_e8m0_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    fp4.load_library()


def _data(seed, M, K, fmt):
    rng = np.random.default_rng(seed)
    x = rng.standard_t(3, (M, K)).astype(np.float32)
    x[:, np.sort(rng.permutation(K)[: K // 64])] *= 100
    xt = torch.from_numpy(x).to(torch.bfloat16)
    return xt, xt.float().numpy()


def _call_noalloc(x, xq, k_hot, out):
    """Straight through the C ABI: no context, no workspace."""
    lib = fp4.load_library()
    op = xq.operand()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fp4_hcp_select_noalloc(ctypes.c_void_p(x.data_ptr()), x.stride(0), ctypes.byref(op), k_hot,
                                      ctypes.c_void_p(out.data_ptr()), st)


OF = {fp4.FP4_FMT_NVFP4: o.NVFP4, fp4.FP4_FMT_MXFP4: o.MXFP4}


def _check_against_oracle(got, ref, xn, xq, fmt, h, label):
    """Both sets ascending; they may differ only within the tie band of the
    oracle's errors (1e-5 relative around the h-th largest)."""
    assert np.all(np.diff(got) > 0), f"{label}: not ascending/distinct"
    c, s, g = o.quantize(xn, OF[fmt])
    e = o.hcp_channel_errors(xn, c, s, OF[fmt], g)
    kth = np.sort(e)[::-1][h - 1]
    diff = set(got.tolist()) ^ set(ref.tolist())
    assert all(abs(e[i] - kth) <= 1e-5 * kth for i in diff), f"{label}: differs outside the tie band"


@pytest.mark.parametrize("fmt", [fp4.FP4_FMT_NVFP4, fp4.FP4_FMT_MXFP4])
@pytest.mark.parametrize("sf_layout", [fp4.FP4_SF_ROWMAJOR, fp4.FP4_SF_MMA])
def test_noalloc_select_matches_workspace_select_twice(fmt, sf_layout):
    """Two calls in a row (the second has fewer channels, then a third on a
    side stream with more), each against fp4_hcp_select and the oracle."""
    for call, (seed, M, K, side) in enumerate([(11, 384, 2048, False), (12, 200, 1024, False),
                                               (13, 96, 1536, True)]):
        xt, xn = _data(seed, M, K, fmt)
        x = xt.cuda()
        h = fp4.fp4_hcp_num_hot(K)
        xq = fp4.fp4_quantize(x, fp4.quant_params(fmt, sf_layout=sf_layout))
        ref = fp4.fp4_hcp_select(x, xq, h).cpu().numpy()
        out = torch.full((h,), -1, dtype=torch.int32, device="cuda")
        if side:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                assert _call_noalloc(x, xq, h, out) == fp4.FP4_OK
            s.synchronize()
        else:
            assert _call_noalloc(x, xq, h, out) == fp4.FP4_OK
            torch.cuda.synchronize()
        _check_against_oracle(out.cpu().numpy(), ref, xn, xq, fmt, h, f"call {call}")


def test_noalloc_empty_rows_and_no_hot_channels_as_workspace_select():
    """rows == 0: both entry points select channels 0..k_hot-1 (every error is 0,
    ties to the lower index); k_hot == 0: both return without writing."""
    K, h = 512, 40
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    xq = fp4.fp4_quantize(x, fp4.quant_params(fp4.FP4_FMT_NVFP4))
    ref = fp4.fp4_hcp_select(x, xq, h).cpu().numpy()
    out = torch.full((h,), -1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(x, xq, h, out) == fp4.FP4_OK
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref) and np.array_equal(ref, np.arange(h))
    xt, _ = _data(14, 64, K, fp4.FP4_FMT_NVFP4)
    xq = fp4.fp4_quantize(xt.cuda(), fp4.quant_params(fp4.FP4_FMT_NVFP4))
    out = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    assert _call_noalloc(xt.cuda(), xq, 0, out) == fp4.FP4_OK
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [-7] * 4


def test_noalloc_rejects_more_channels_than_its_scratch():
    K = fp4.FP4_NOALLOC_MAX_CHANNELS + 32
    x = torch.zeros((16, K), dtype=torch.bfloat16, device="cuda")
    xq = fp4.fp4_quantize(x, fp4.quant_params(fp4.FP4_FMT_MXFP4))
    out = torch.zeros((8,), dtype=torch.int32, device="cuda")
    assert _call_noalloc(x, xq, 8, out) == fp4.FP4_ERR_TOO_LARGE
