"""Block-scaled FP4 (MXFP4 / NVFP4) quantization and GEMMs for GB300 (sm_103a).

A thin ctypes binding over the C ABI declared in ``include/fp4.h``; every step
of the computation runs in the library's CUDA kernels.  PyTorch supplies
device memory and the current stream.  The functions carry the C names;
outputs that are not passed in are allocated with ``torch.empty``.

There is no CPU fallback: if the shared library has not been built, or no GPU
is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

import torch

from .build import lib_path

# ---- constants (mirror include/fp4.h) ---------------------------------------
(FP4_OK, FP4_ERR_INVALID_ARG, FP4_ERR_UNSUPPORTED, FP4_ERR_MISALIGNED, FP4_ERR_CUDA, FP4_ERR_TIMEOUT,
 FP4_ERR_TOO_LARGE) = range(7)
FP4_NOALLOC_MAX_CHANNELS = 65536
FP4_FMT_MXFP4, FP4_FMT_NVFP4 = 0, 1
FP4_ROUND_RTN, FP4_ROUND_SR = 0, 1
FP4_SCALING_1D, FP4_SCALING_2D = 0, 1
FP4_SF_ROWMAJOR, FP4_SF_MMA = 0, 1
FP4_DTYPE_BF16, FP4_DTYPE_F32 = 0, 1
FP4_HCP_SINGLE, FP4_HCP_TWO, FP4_HCP_TWO_FP8, FP4_HCP_SINGLE_MXFP8 = 0, 1, 2, 3
BLOCK = {FP4_FMT_MXFP4: 32, FP4_FMT_NVFP4: 16}


class FP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fp4_status_string(status)} (status {status})")


class fp4_quant_params(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("block", ctypes.c_int32), ("rounding", ctypes.c_int32),
                ("scaling", ctypes.c_int32), ("transpose", ctypes.c_int32), ("rht", ctypes.c_int32),
                ("sf_layout", ctypes.c_int32), ("sr_stream", ctypes.c_uint32), ("sr_seed", ctypes.c_uint64),
                ("sr_offset", ctypes.c_uint64), ("rht_seed", ctypes.c_uint64)]


class fp4_operand(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p),
                ("format", ctypes.c_int32), ("sf_layout", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("k", ctypes.c_int64), ("block", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32, _I64, _U64, _F32, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "fp4_create": (ctypes.c_int, [ctypes.POINTER(_P)]),
    "fp4_destroy": (None, [_P]),
    "fp4_sync_status": (ctypes.c_int, [_P, _P]),
    "fp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fp4_scales_bytes": (_SZ, [_I64, _I64, _I32, _I32, _I32]),
    "fp4_amax": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I64, _I32, _U64, _P, _P]),
    "fp4_quantize": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I64, ctypes.POINTER(fp4_quant_params), _P, _P, _P,
                                    _P, _P]),
    "fp4_quantize_dual": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I64, ctypes.POINTER(fp4_quant_params),
                                         ctypes.POINTER(fp4_quant_params), _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "fp4_dequantize": (ctypes.c_int, [_P, ctypes.POINTER(fp4_operand), _I32, _P, _I64, _P]),
    "fp4_rht16": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I64, _I32, _U64, _P, _P]),
    "fp4_dge_backward": (ctypes.c_int, [_P, _P, _I32, _I64, ctypes.POINTER(fp4_operand), _P, _I32, _I64, _P, _I64,
                                        _F32, _F32, _F32, _P]),
    "fp4_soft_forward": (ctypes.c_int, [_P, _P, _I32, _I64, ctypes.POINTER(fp4_operand), _P, _I64, _F32, _P]),
    "fp4_soft_backward": (ctypes.c_int, [_P, _P, _I32, _I64, ctypes.POINTER(fp4_operand), _P, _I32, _I64, _P, _I64,
                                         _F32, _P]),
    "fp4_occ_threshold_workspace_bytes": (_SZ, [_I32]),
    "fp4_occ_max_outliers": (_I64, [_I64, _I64, ctypes.c_double]),
    "fp4_occ_threshold": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I64, ctypes.c_double, _P, _P, _P, _SZ, _P]),
    "fp4_occ_quantize": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I64, ctypes.POINTER(fp4_quant_params), _P, _P, _P,
                                        _P, _P, _P]),
    "fp4_occ_gemm_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I32, _I64]),
    "fp4_occ_gemm": (ctypes.c_int, [_P, _P, _I32, _I64, _P, _I64, ctypes.POINTER(fp4_operand),
                                    ctypes.POINTER(fp4_operand), _P, _P, _I32, _I64, _I32, _P, _I64, _P, _SZ, _P]),
    "fp4_quant_error_stats": (ctypes.c_int, [_P, _P, _I32, _I64, ctypes.POINTER(fp4_operand), _P, _F32, _P, _P, _P]),
    "fp4_gemm": (ctypes.c_int, [_P, ctypes.POINTER(fp4_operand), ctypes.POINTER(fp4_operand), _I32, _P, _I64, _I32,
                                _P]),
    "fp4_gemm_quant_a": (ctypes.c_int, [_P, _P, _I64, _I64, ctypes.POINTER(fp4_operand), _I32, _P, _I64, _P, _P,
                                        _P]),
    "fp4_hcp_num_hot": (_I32, [_I64, ctypes.c_double]),
    "fp4_hcp_select_workspace_bytes": (_SZ, [_I64]),
    "fp4_hcp_select": (ctypes.c_int, [_P, _P, _I64, ctypes.POINTER(fp4_operand), _I32, _P, _P, _SZ, _P]),
    "fp4_hcp_select_noalloc": (ctypes.c_int, [_P, _I64, ctypes.POINTER(fp4_operand), _I32, _P, _P]),
    "fp4_hcp_workspace_bytes": (_SZ, [_I64, _I64, _I32, _I32]),
    "fp4_hcp_quantize_zeroed": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I64, ctypes.POINTER(fp4_quant_params), _P,
                                               _I32, _P, _P, _P, _P]),
    "fp4_hcp_gemm": (ctypes.c_int, [_P, _P, _I64, _P, _I64, ctypes.POINTER(fp4_operand),
                                    ctypes.POINTER(fp4_operand), _P, _I32, _I32, _I32, _P, _SZ, _I32, _P, _I64, _P]),
    "fp4_encode_e2m1": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _P]),
    "fp4_encode_e4m3": (ctypes.c_int, [_P, _P, _P, _I64, _P]),
}

_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with fp4_block_scaled_e8m0_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == lib_path():
        _lib = lib
    return lib


def declared_symbols(header: Optional[str] = None) -> list[str]:
    """Names of the functions include/fp4.h declares."""
    header = header or os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fp4.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4_[a-z0-9_]+)\s*\(", text)))


def _check(status: int, where: str) -> None:
    if status != FP4_OK:
        raise FP4Error(status, where)


def fp4_status_string(status: int) -> str:
    try:
        return load_library().fp4_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


def fp4_scales_bytes(rows: int, k: int, fmt: int, sf_layout: int, block: int = 0) -> int:
    return int(load_library().fp4_scales_bytes(rows, k, fmt, sf_layout, block))


# ---- context ----------------------------------------------------------------
class Context:
    """Owns an fp4_ctx (device scratch for one stream at a time)."""

    def __init__(self):
        self._lib = load_library()
        h = _P()
        _check(self._lib.fp4_create(ctypes.byref(h)), "fp4_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self._lib.fp4_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_contexts: dict[int, Context] = {}


def fp4_create() -> Context:
    return Context()


def fp4_destroy(ctx: Context) -> None:
    ctx.close()


def default_context() -> Context:
    dev = torch.cuda.current_device()
    if dev not in _contexts:
        _contexts[dev] = Context()
    return _contexts[dev]


def _ctx(ctx):
    return (ctx or default_context()).handle


def _stream(stream) -> _P:
    if stream is None:
        stream = torch.cuda.current_stream()
    return _P(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def fp4_sync_status(ctx: Optional[Context] = None, stream=None) -> int:
    """Synchronize the stream and return the context's device status (0 = ok)."""
    return load_library().fp4_sync_status(_ctx(ctx), _stream(stream))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else _P(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FP4_DTYPE_BF16
    if t.dtype == torch.float32:
        return FP4_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ld(t: torch.Tensor) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


# ---- quantized tensor ---------------------------------------------------------
@dataclass
class QTensor:
    """A quantized operand: rows x k values, blocks along k."""
    codes: torch.Tensor                # uint8 [rows, k/2]
    scales: torch.Tensor               # uint8, layout sf_layout
    tensor_scale: Optional[torch.Tensor]  # float32 [1] (NVFP4)
    fmt: int
    sf_layout: int
    rows: int
    k: int
    block: int = 0                     # elements per scale; 0 = the format's own

    def operand(self) -> fp4_operand:
        return fp4_operand(self.codes.data_ptr(), self.scales.data_ptr(),
                           self.tensor_scale.data_ptr() if self.tensor_scale is not None else None,
                           self.fmt, self.sf_layout, self.rows, self.k, self.block)


def quant_params(fmt=FP4_FMT_NVFP4, rounding=FP4_ROUND_RTN, scaling=FP4_SCALING_1D, transpose=False, rht=False,
                 sf_layout=FP4_SF_MMA, sr_seed=0, sr_offset=0, sr_stream=0, rht_seed=0,
                 block: int = 0) -> fp4_quant_params:
    return fp4_quant_params(fmt, block or BLOCK[fmt], rounding, scaling, int(transpose), int(rht), sf_layout,
                            sr_stream, sr_seed, sr_offset, rht_seed)


def alloc_qtensor(rows: int, k: int, fmt: int, sf_layout: int, device, block: int = 0) -> QTensor:
    block = 0 if block == BLOCK[fmt] else block
    sb = fp4_scales_bytes(rows, k, fmt, sf_layout, block)
    return QTensor(torch.empty((rows, k // 2), dtype=torch.uint8, device=device),
                   torch.empty((max(sb, 1),), dtype=torch.uint8, device=device),
                   torch.empty((1,), dtype=torch.float32, device=device) if fmt == FP4_FMT_NVFP4 else None,
                   fmt, sf_layout, rows, k, block)


def fp4_amax(x: torch.Tensor, rht_axis: int = -1, rht_seed: int = 0, out: Optional[torch.Tensor] = None,
             ctx=None, stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty((1,), dtype=torch.float32, device=x.device)
    _check(load_library().fp4_amax(_ctx(ctx), _ptr(x), _dtype_code(x), x.shape[0], x.shape[1], _ld(x), rht_axis,
                                   rht_seed, _ptr(out), _stream(stream)), "fp4_amax")
    return out


def fp4_quantize(x: torch.Tensor, params: fp4_quant_params, given_amax: Optional[torch.Tensor] = None,
                 out: Optional[QTensor] = None, ctx=None, stream=None) -> QTensor:
    rows, cols = x.shape
    o_rows, blocked = (cols, rows) if params.transpose else (rows, cols)
    out = out or alloc_qtensor(o_rows, blocked, params.format, params.sf_layout, x.device, params.block)
    _check(load_library().fp4_quantize(_ctx(ctx), _ptr(x), _dtype_code(x), rows, cols, _ld(x), ctypes.byref(params),
                                       _ptr(given_amax), _ptr(out.codes), _ptr(out.scales), _ptr(out.tensor_scale),
                                       _stream(stream)), "fp4_quantize")
    return out


def fp4_quantize_dual(x: torch.Tensor, p_rows: fp4_quant_params, p_cols: fp4_quant_params,
                      given_amax_rows=None, given_amax_cols=None, out_rows: Optional[QTensor] = None,
                      out_cols: Optional[QTensor] = None, ctx=None, stream=None):
    rows, cols = x.shape
    out_rows = out_rows or alloc_qtensor(rows, cols, p_rows.format, p_rows.sf_layout, x.device)
    out_cols = out_cols or alloc_qtensor(cols, rows, p_cols.format, p_cols.sf_layout, x.device)
    _check(load_library().fp4_quantize_dual(
        _ctx(ctx), _ptr(x), _dtype_code(x), rows, cols, _ld(x), ctypes.byref(p_rows), ctypes.byref(p_cols),
        _ptr(given_amax_rows), _ptr(given_amax_cols), _ptr(out_rows.codes), _ptr(out_rows.scales),
        _ptr(out_rows.tensor_scale), _ptr(out_cols.codes), _ptr(out_cols.scales), _ptr(out_cols.tensor_scale),
        _stream(stream)), "fp4_quantize_dual")
    return out_rows, out_cols


def fp4_dequantize(q: QTensor, out_dtype=torch.float32, out: Optional[torch.Tensor] = None, ctx=None,
                   stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty((q.rows, q.k), dtype=out_dtype, device=q.codes.device)
    op = q.operand()
    _check(load_library().fp4_dequantize(_ctx(ctx), ctypes.byref(op), _dtype_code(out), _ptr(out), _ld(out),
                                         _stream(stream)), "fp4_dequantize")
    return out


def fp4_rht16(x: torch.Tensor, axis: int, seed: int, out: Optional[torch.Tensor] = None, ctx=None,
              stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty(x.shape, dtype=torch.float32, device=x.device)
    _check(load_library().fp4_rht16(_ctx(ctx), _ptr(x), _dtype_code(x), x.shape[0], x.shape[1], _ld(x), axis, seed,
                                     _ptr(out), _stream(stream)), "fp4_rht16")
    return out


def fp4_dge_backward(x: torch.Tensor, q: QTensor, dy: torch.Tensor, k: float = 5.0, clamp: float = 3.0,
                     outside: float = 1.0, out: Optional[torch.Tensor] = None, ctx=None, stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty(x.shape, dtype=torch.float32, device=x.device)
    op = q.operand()
    _check(load_library().fp4_dge_backward(_ctx(ctx), _ptr(x), _dtype_code(x), _ld(x), ctypes.byref(op), _ptr(dy),
                                           _dtype_code(dy), _ld(dy), _ptr(out), _ld(out), k, clamp, outside,
                                           _stream(stream)), "fp4_dge_backward")
    return out


def fp4_soft_forward(x: torch.Tensor, q: QTensor, beta: float, out: Optional[torch.Tensor] = None, ctx=None,
                     stream=None) -> torch.Tensor:
    """y = s Q_soft(x / s), fp32 (sigmoid-smoothed quantizer)."""
    out = out if out is not None else torch.empty(x.shape, dtype=torch.float32, device=x.device)
    op = q.operand()
    _check(load_library().fp4_soft_forward(_ctx(ctx), _ptr(x), _dtype_code(x), _ld(x), ctypes.byref(op), _ptr(out),
                                           _ld(out), beta, _stream(stream)), "fp4_soft_forward")
    return out


def fp4_soft_backward(x: torch.Tensor, q: QTensor, dy: torch.Tensor, beta: float, out: Optional[torch.Tensor] = None,
                      ctx=None, stream=None) -> torch.Tensor:
    """dx = dy Q_soft'(x / s), fp32 (sigmoid-smoothed estimator)."""
    out = out if out is not None else torch.empty(x.shape, dtype=torch.float32, device=x.device)
    op = q.operand()
    _check(load_library().fp4_soft_backward(_ctx(ctx), _ptr(x), _dtype_code(x), _ld(x), ctypes.byref(op), _ptr(dy),
                                            _dtype_code(dy), _ld(dy), _ptr(out), _ld(out), beta, _stream(stream)),
           "fp4_soft_backward")
    return out


def fp4_gemm(a: QTensor, b: QTensor, out_dtype=torch.bfloat16, out: Optional[torch.Tensor] = None,
             accumulate: bool = False, ctx=None, stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty((a.rows, b.rows), dtype=out_dtype, device=a.codes.device)
    oa, ob = a.operand(), b.operand()
    _check(load_library().fp4_gemm(_ctx(ctx), ctypes.byref(oa), ctypes.byref(ob), _dtype_code(out), _ptr(out),
                                   _ld(out), int(accumulate), _stream(stream)), "fp4_gemm")
    return out


def fp4_gemm_quant_a(x: torch.Tensor, b: QTensor, out_dtype=torch.bfloat16, out: Optional[torch.Tensor] = None,
                     a_out: Optional[QTensor] = None, ctx=None, stream=None) -> torch.Tensor:
    """C = Q(x) b^T with x (bf16) quantized to MXFP4 (RTN, 1D) inside the GEMM.

    a_out (an MXFP4 QTensor in the MMA scale layout, e.g. from alloc_qtensor)
    also receives x's quantization."""
    m = x.shape[0]
    out = out if out is not None else torch.empty((m, b.rows), dtype=out_dtype, device=x.device)
    ob = b.operand()
    _check(load_library().fp4_gemm_quant_a(_ctx(ctx), _ptr(x), m, _ld(x), ctypes.byref(ob), _dtype_code(out),
                                           _ptr(out), _ld(out), _ptr(a_out.codes if a_out else None),
                                           _ptr(a_out.scales if a_out else None), _stream(stream)),
           "fp4_gemm_quant_a")
    return out


def fp4_hcp_num_hot(k: int, ratio: float = 0.09) -> int:
    """h = ceil(ratio * K), computed by the library: the "top 9%" channel count."""
    h = int(load_library().fp4_hcp_num_hot(k, ratio))
    if h < 0:
        raise ValueError(f"fp4_hcp_num_hot: k = {k}, ratio = {ratio} outside k >= 0, 0 <= ratio <= 1")
    return h


def fp4_hcp_select(x: torch.Tensor, xq: QTensor, k_hot: int, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, ctx=None, stream=None) -> torch.Tensor:
    lib = load_library()
    out = out if out is not None else torch.empty((max(k_hot, 1),), dtype=torch.int32, device=x.device)
    ws_bytes = int(lib.fp4_hcp_select_workspace_bytes(xq.k))
    workspace = workspace if workspace is not None else torch.empty((max(ws_bytes, 1),), dtype=torch.uint8,
                                                                   device=x.device)
    op = xq.operand()
    _check(lib.fp4_hcp_select(_ctx(ctx), _ptr(x), _ld(x), ctypes.byref(op), k_hot, _ptr(out), _ptr(workspace),
                              workspace.numel(), _stream(stream)), "fp4_hcp_select")
    return out[:k_hot]


def fp4_hcp_select_noalloc(x: torch.Tensor, xq: QTensor, k_hot: int, out: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """Hot-channel selection without a context or workspace.

    For callers that may not allocate device memory (their memory belongs to
    their own caching pool, or they cannot afford the synchronization that
    cudaMalloc/cudaFree may cause): the library keeps a fixed scratch array for
    up to FP4_NOALLOC_MAX_CHANNELS channels.  Calls that overlap on the GPU
    race; the first call on a device should come before any stream capture.
    `out` (int32[k_hot]) must be given by a caller that may not allocate.
    """
    out = out if out is not None else torch.empty((max(k_hot, 1),), dtype=torch.int32, device=x.device)
    op = xq.operand()
    _check(load_library().fp4_hcp_select_noalloc(_ptr(x), _ld(x), ctypes.byref(op), k_hot, _ptr(out),
                                                 _stream(stream)), "fp4_hcp_select_noalloc")
    return out[:k_hot]


def fp4_hcp_quantize_zeroed(x: torch.Tensor, params: fp4_quant_params, hot_idx: torch.Tensor, k_hot: int,
                            out: Optional[QTensor] = None, ctx=None, stream=None) -> QTensor:
    """Quantize x with the hot channels (ascending int32 list) set to zero: the operand of the order-0 HCP GEMM."""
    rows, cols = x.shape
    out = out or alloc_qtensor(rows, cols, params.format, params.sf_layout, x.device)
    _check(load_library().fp4_hcp_quantize_zeroed(_ctx(ctx), _ptr(x), _dtype_code(x), rows, cols, _ld(x),
                                                  ctypes.byref(params), _ptr(hot_idx), k_hot, _ptr(out.codes),
                                                  _ptr(out.scales), _ptr(out.tensor_scale), _stream(stream)),
           "fp4_hcp_quantize_zeroed")
    return out


def fp4_hcp_gemm(x: torch.Tensor, w: torch.Tensor, xq: QTensor, wq: QTensor, hot_idx: torch.Tensor, k_hot: int,
                 mode: int = FP4_HCP_SINGLE, order: int = 2, out_dtype=torch.bfloat16,
                 out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, ctx=None,
                 stream=None) -> torch.Tensor:
    lib = load_library()
    out = out if out is not None else torch.empty((xq.rows, wq.rows), dtype=out_dtype, device=x.device)
    ws_bytes = int(lib.fp4_hcp_workspace_bytes(xq.rows, wq.rows, k_hot, order))
    workspace = workspace if workspace is not None else torch.empty((max(ws_bytes, 1),), dtype=torch.uint8,
                                                                   device=x.device)
    ox, ow = xq.operand(), wq.operand()
    _check(lib.fp4_hcp_gemm(_ctx(ctx), _ptr(x), _ld(x), _ptr(w), _ld(w), ctypes.byref(ox), ctypes.byref(ow),
                            _ptr(hot_idx), k_hot, mode, order, _ptr(workspace), workspace.numel(), _dtype_code(out),
                            _ptr(out), _ld(out), _stream(stream)), "fp4_hcp_gemm")
    return out


# ---- outlier clamping and compensation ----------------------------------------
def fp4_occ_max_outliers(rows: int, cols: int, q: float = 0.99) -> int:
    return int(load_library().fp4_occ_max_outliers(rows, cols, q))


def fp4_occ_threshold(x: torch.Tensor, q: float = 0.99, workspace: Optional[torch.Tensor] = None, ctx=None,
                      stream=None):
    """(tau, n_outliers): device fp32[1] and int64[1]."""
    lib = load_library()
    tau = torch.empty((1,), dtype=torch.float32, device=x.device)
    n_out = torch.empty((1,), dtype=torch.int64, device=x.device)
    ws_bytes = int(lib.fp4_occ_threshold_workspace_bytes(_dtype_code(x)))
    workspace = workspace if workspace is not None else torch.empty((ws_bytes,), dtype=torch.uint8, device=x.device)
    _check(lib.fp4_occ_threshold(_ctx(ctx), _ptr(x), _dtype_code(x), x.shape[0], x.shape[1], _ld(x), q, _ptr(tau),
                                 _ptr(n_out), _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4_occ_threshold")
    return tau, n_out


def fp4_occ_quantize(x: torch.Tensor, params: fp4_quant_params, tau: torch.Tensor, out: Optional[QTensor] = None,
                     col_counts: Optional[torch.Tensor] = None, ctx=None, stream=None) -> QTensor:
    """Quantize clamp(x, -tau, tau) in the row layout; col_counts (float32[cols]) gets the outliers per column."""
    rows, cols = x.shape
    out = out or alloc_qtensor(rows, cols, params.format, params.sf_layout, x.device)
    _check(load_library().fp4_occ_quantize(_ctx(ctx), _ptr(x), _dtype_code(x), rows, cols, _ld(x),
                                           ctypes.byref(params), _ptr(tau), _ptr(out.codes), _ptr(out.scales),
                                           _ptr(out.tensor_scale), _ptr(col_counts), _stream(stream)),
           "fp4_occ_quantize")
    return out


def fp4_occ_gemm(x: torch.Tensor, w: torch.Tensor, xq: QTensor, wq: QTensor, tau: torch.Tensor,
                 col_counts: Optional[torch.Tensor], k_dense: int, max_outliers: int, out_dtype=torch.bfloat16,
                 out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, ctx=None,
                 stream=None) -> torch.Tensor:
    """Y = alpha Q(X_c) Q(W)^T + dX W^T."""
    lib = load_library()
    out = out if out is not None else torch.empty((xq.rows, wq.rows), dtype=out_dtype, device=x.device)
    ws_bytes = int(lib.fp4_occ_gemm_workspace_bytes(xq.rows, wq.rows, xq.k, k_dense, max_outliers))
    workspace = workspace if workspace is not None else torch.empty((max(ws_bytes, 1),), dtype=torch.uint8,
                                                                   device=x.device)
    ox, ow = xq.operand(), wq.operand()
    _check(lib.fp4_occ_gemm(_ctx(ctx), _ptr(x), _dtype_code(x), _ld(x), _ptr(w), _ld(w), ctypes.byref(ox),
                            ctypes.byref(ow), _ptr(tau), _ptr(col_counts), k_dense, max_outliers, _dtype_code(out),
                            _ptr(out), _ld(out), _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4_occ_gemm")
    return out


STAT_NAMES = ("cos", "mse", "snr_db", "rel_err")


def fp4_quant_error_stats(x: torch.Tensor, q: QTensor, tau: Optional[torch.Tensor] = None, beta: float = 0.0,
                          ctx=None, stream=None):
    """(sums, stats), device float64[4] each.  sums: sum x^2, sum x_hat^2, sum x x_hat,
    sum (x - x_hat)^2 (x_hat: the dequantized value, + the clamped-away part with tau, or
    s Q_soft(x/s) with beta > 0).  stats: cosine, MSE, SNR (dB), relative L2 error, formed by
    the library from the sums (names in STAT_NAMES)."""
    sums = torch.empty((4,), dtype=torch.float64, device=x.device)
    stats = torch.empty((4,), dtype=torch.float64, device=x.device)
    op = q.operand()
    _check(load_library().fp4_quant_error_stats(_ctx(ctx), _ptr(x), _dtype_code(x), _ld(x), ctypes.byref(op),
                                                _ptr(tau), beta, _ptr(sums), _ptr(stats), _stream(stream)),
           "fp4_quant_error_stats")
    return sums, stats


def stats_dict(stats) -> dict:
    """The four quality numbers by name (no arithmetic)."""
    return {name: float(v) for name, v in zip(STAT_NAMES, stats)}


def fp4_encode_e2m1(xs: torch.Tensor, method: int = 0, ctx=None, stream=None) -> torch.Tensor:
    out = torch.empty(xs.shape, dtype=torch.uint8, device=xs.device)
    _check(load_library().fp4_encode_e2m1(_ctx(ctx), _ptr(xs), _ptr(out), xs.numel(), method, _stream(stream)),
           "fp4_encode_e2m1")
    return out


def fp4_encode_e4m3(t: torch.Tensor, ctx=None, stream=None) -> torch.Tensor:
    out = torch.empty(t.shape, dtype=torch.uint8, device=t.device)
    _check(load_library().fp4_encode_e4m3(_ctx(ctx), _ptr(t), _ptr(out), t.numel(), _stream(stream)),
           "fp4_encode_e4m3")
    return out
