#!/usr/bin/env python
"""Benchmark of the block-scaled FP4 hot path on one LLaMA-1B-shaped linear layer.

One step = the forward and backward pass of the MLP up-projection
Y[M,N] = X[M,K] W[N,K]^T with M = 8192 tokens, K = 2048, N = 5632 in NVFP4:

  forward   quantize X and W, each in both layouts from one read: the forward
            layout (RTN, 1D blocks of 16 along K, E4M3 scale x per-tensor fp32
            scale) and the backward one (transposed, SR + RHT16 along the
            blocked axis; 16x16 2D blocks for W); fprop GEMM Y = Xq Wq^T (bf16)
  backward  quantize dY in both layouts from one read (SR + RHT16 along N for
            dgrad, along M for wgrad); dgrad GEMM dX = dYq Wq_t^T (bf16),
            wgrad GEMM dW = dYq_m Xq_t^T (fp32); DGE backward
            dW' = dW * f'(W / s_W) (k = 5, clamp 3.0)

Independent ops run on two streams: the W quantization beside the X one, and
wgrad + DGE beside dgrad (each op waits for what it reads).  The per-op
breakdown times every op alone.

Every step runs in the library's CUDA kernels through the C ABI.  Inputs are
seeded synthetic tensors (X ~ N(0,1), W ~ N(0,0.02), dY ~ N(0,1e-3)) resident
in HBM before the timed region; L2 is flushed (512 MiB write) before each
timed step.  Prints one JSON line (see the keys below).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP4 quantize GB/s and block-scaled FP4 GEMM TFLOP/s, % of GB300 roofline"
M, K, N = 8192, 2048, 5632
GEMM_FLOPS = 2 * M * N * K          # per GEMM; three per step
STEP_FLOPS = 3 * GEMM_FLOPS
FP4_OVER_BF16 = 13.5 / 2.25         # nominal dense FP4 : BF16 tensor rate
WORKLOAD = ("llama1b_mlp_up fwd+bwd: X[8192,2048] W[5632,2048] dY[8192,5632] bf16; NVFP4; fwd RTN 1D, "
            "bwd SR + RHT16 (+16x16 2D on W); each of X, W, dY quantized in both layouts from one read; "
            "fprop/dgrad/wgrad GEMMs; DGE (k=5, clamp 3) on W")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", default="512x704", help="MxN rows of the CPU-baseline sample (K stays 2048)")
    ap.add_argument("--ext-launches", type=int, default=20,
                    help="timed launches of each op outside the step (0: skip them)")
    ap.add_argument("--ext-only", action="store_true",
                    help="run only the ops outside the step (one warm-up step first) and print their JSON")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic bytes per element of each op (one read of inputs + writes)
# ---------------------------------------------------------------------------
DUAL_Q_BYTES = 2 + 2 * (0.5 + 1 / 16)  # bf16 in once; codes + E4M3 bytes for both layouts
OPS = {
    #  name           kind     units per launch (bytes or flops)
    "quant_x_dual":  ("hbm", M * K * DUAL_Q_BYTES),
    "quant_w_dual":  ("hbm", N * K * DUAL_Q_BYTES),
    "fprop":         ("tensor", GEMM_FLOPS),
    "quant_dy_dual": ("hbm", M * N * DUAL_Q_BYTES),
    "dgrad":         ("tensor", GEMM_FLOPS),
    "wgrad":         ("tensor", GEMM_FLOPS),
    "dge":           ("hbm", N * K * (2 + 4 + 4) + N * K / 16),
}
# our kernels per op: amax (both layouts) + quantize (both layouts) for each dual
KERNELS_PER_OP = {"quant_x_dual": 2, "quant_w_dual": 2, "fprop": 1, "quant_dy_dual": 2, "dgrad": 1, "wgrad": 1,
                  "dge": 1}


class Step:
    """Buffers and calls of one fwd+bwd step (all device-resident).

    The step's ops form a small dependency graph.  The forward quantizes X and
    W independently; the backward's dgrad and wgrad are independent, and the
    DGE scales wgrad's output.  With a side stream, `run` puts the ops in SIDE
    there (with a context of their own: a context serves one stream at a time)
    and makes each op wait for the ones it reads on the other stream (WAITS),
    so that one op's last partial wave overlaps the other's work."""

    SIDE = ("quant_w_dual", "wgrad", "dge")
    WAITS = {"fprop": "quant_w_dual", "wgrad": "quant_dy_dual"}

    def __init__(self, fp4, X, W, dY, dev):
        self.fp4 = fp4
        self.side_ctx = fp4.Context()
        self.X, self.W, self.dY = X, W, dY
        NV, SR, T2D = fp4.FP4_FMT_NVFP4, fp4.FP4_ROUND_SR, fp4.FP4_SCALING_2D
        self.p_fwd = fp4.quant_params(NV)
        self.p_dy_n = fp4.quant_params(NV, SR, rht=True, sr_seed=2, sr_stream=0, rht_seed=2)
        self.p_w_t = fp4.quant_params(NV, SR, T2D, transpose=True, rht=True, sr_seed=2, sr_stream=1, rht_seed=2)
        self.p_dy_m = fp4.quant_params(NV, SR, transpose=True, rht=True, sr_seed=2, sr_stream=2, rht_seed=2)
        self.p_x_t = fp4.quant_params(NV, SR, transpose=True, rht=True, sr_seed=2, sr_stream=3, rht_seed=2)
        a = fp4.alloc_qtensor
        self.xq = a(M, K, NV, fp4.FP4_SF_MMA, dev)
        self.wq = a(N, K, NV, fp4.FP4_SF_MMA, dev)
        self.dyq_n = a(M, N, NV, fp4.FP4_SF_MMA, dev)
        self.dyq_m = a(N, M, NV, fp4.FP4_SF_MMA, dev)
        self.wq_t = a(K, N, NV, fp4.FP4_SF_MMA, dev)
        self.xq_t = a(K, M, NV, fp4.FP4_SF_MMA, dev)
        self.Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty((N, K), dtype=torch.float32, device=dev)
        self.dWd = torch.empty((N, K), dtype=torch.float32, device=dev)

    def ops(self, step_idx: int, side_ctx=None):
        f = self.fp4
        off = step_idx << 40      # a fresh SR draw every step
        for p in (self.p_dy_n, self.p_w_t, self.p_dy_m, self.p_x_t):
            p.sr_offset = off
        sc = side_ctx
        return [
            ("quant_x_dual", lambda: f.fp4_quantize_dual(self.X, self.p_fwd, self.p_x_t, out_rows=self.xq,
                                                         out_cols=self.xq_t)),
            ("quant_w_dual", lambda: f.fp4_quantize_dual(self.W, self.p_fwd, self.p_w_t, out_rows=self.wq,
                                                         out_cols=self.wq_t, ctx=sc)),
            ("fprop", lambda: f.fp4_gemm(self.xq, self.wq, out=self.Y)),
            ("quant_dy_dual", lambda: f.fp4_quantize_dual(self.dY, self.p_dy_n, self.p_dy_m, out_rows=self.dyq_n,
                                                          out_cols=self.dyq_m)),
            ("dgrad", lambda: f.fp4_gemm(self.dyq_n, self.wq_t, out=self.dX)),
            ("wgrad", lambda: f.fp4_gemm(self.dyq_m, self.xq_t, out=self.dW, ctx=sc)),
            ("dge", lambda: f.fp4_dge_backward(self.W, self.wq, self.dW, 5.0, 3.0, 1.0, out=self.dWd, ctx=sc)),
        ]

    def run(self, step_idx: int, events=None, before=None, after=None, side=None):
        """Enqueue the step's ops: all on the current stream in order, or, with a
        `side` stream, the SIDE ops there (the step still starts after, and
        ends before, what the current stream holds around it).  `before`/`after`
        map an op name to a callable taking the op's stream, run just before /
        after the op is enqueued (the end-to-end loop uses them to wait for
        inputs and to start copies); `events` brackets each op."""
        main = torch.cuda.current_stream()
        if side is not None:
            side.wait_stream(main)
        done = {}
        for name, fn in self.ops(step_idx, self.side_ctx if side is not None else None):
            s = side if side is not None and name in self.SIDE else main
            if side is not None and name in self.WAITS:
                s.wait_event(done[self.WAITS[name]])
            with torch.cuda.stream(s):
                if before and name in before:
                    before[name](s)
                if events is not None:
                    events[name][0].record(s)
                fn()
                if events is not None:
                    events[name][1].record(s)
                if after and name in after:
                    after[name](s)
            if side is not None:
                done[name] = torch.cuda.Event()
                done[name].record(s)
        if side is not None:
            main.wait_stream(side)


# ---------------------------------------------------------------------------
# ops outside the step, on the step's tensors: the sigmoid-smoothed estimator
# (an alternative to the DGE backward on W, "深度学习中的梯度计算基础" §3.2)
# ---------------------------------------------------------------------------
SOFT_BWD_BYTES = N * K * (2 + 4 + 4) + N * K / 16     # W, dW in; dW' out; scales
SOFT_FWD_BYTES = N * K * (2 + 4) + N * K / 16         # W in; s Q_soft(W/s) out; scales


def extension_ops(fp4, step, dev):
    out = torch.empty((N, K), dtype=torch.float32, device=dev)
    ops = []
    for beta in (40.0, 10.0, 1.0):
        ops.append((f"soft_backward_beta{beta:g}", SOFT_BWD_BYTES,
                    lambda b=beta: fp4.fp4_soft_backward(step.W, step.wq, step.dW, b, out=out)))
    for beta in (40.0, 1.0):
        ops.append((f"soft_forward_beta{beta:g}", SOFT_FWD_BYTES,
                    lambda b=beta: fp4.fp4_soft_forward(step.W, step.wq, b, out=out)))
    return ops


def _time_op(fn, flush, launches):
    """Mean device time of `fn` over `launches` calls, L2 flushed before each."""
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    for i in range(launches):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) * 1e-3 for a, b in ev]))


def _rate(kind, units, t, pk):
    if kind == "tensor":
        peak = pk["bf16_tflops_sustained"] * FP4_OVER_BF16
        r = units / t / 1e12
        return {"us": t * 1e6, "rate": r, "unit": "TFLOP/s", "frac": r / peak}
    r = units / t / 1e9
    return {"us": t * 1e6, "rate": r, "unit": "GB/s", "frac": r / pk["hbm_gbs"]}


def time_extensions(fp4, step, dev, flush, launches, pk):
    """Each op timed alone: L2 flushed before every launch, CUDA events around it."""
    res = {}
    for name, nbytes, fn in extension_ops(fp4, step, dev):
        res[name] = dict(_rate("hbm", nbytes, _time_op(fn, flush, launches), pk), launches=launches)
    res["occ"] = time_occ(fp4, dev, flush, launches, pk)
    res["block_sweep"] = block_sweep(fp4, step, dev, flush, launches, pk)
    res["hcp"] = time_hcp(fp4, dev, flush, launches, pk)
    return res


def time_hcp(fp4, dev, flush, launches, pk):
    """Hot-channel compensation ("大模型4位训练中的异常值动态分析与优化实践" §3-4) on the hot-channel
    activations: plain NVFP4 GEMM, order-2 compensation (bf16 residual columns), the variant with
    the hot channels zeroed before quantizing (their product in bf16), single-kernel and with the
    residual as a second GEMM in bf16 or E4M3; h = 9% of K.  Relative L2 error of Y against the
    fp64 product on 64 sampled rows."""
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.hcp_square(OCC_M, OCC_K, OCC_N)
    X, W = d["X"].to(dev), d["W"].to(dev)
    NV = fp4.FP4_FMT_NVFP4
    p = fp4.quant_params(NV)
    xq, wq = fp4.fp4_quantize(X, p), fp4.fp4_quantize(W, p)
    h = fp4.hcp_num_hot(OCC_K)
    hot = fp4.fp4_hcp_select(X, xq, h)
    x0q = fp4.fp4_hcp_quantize_zeroed(X, p, hot, h)
    lib = fp4.load_library()
    ws = torch.empty((max(lib.fp4_hcp_workspace_bytes(OCC_M, OCC_N, h, 2), 1),), dtype=torch.uint8, device=dev)
    Y = torch.empty((OCC_M, OCC_N), dtype=torch.bfloat16, device=dev)
    flops = 2 * OCC_M * OCC_N * OCC_K
    rows = np.random.default_rng(0).choice(OCC_M, 64, replace=False)
    exact = d["X"].float().numpy()[rows].astype(np.float64) @ d["W"].float().numpy().astype(np.float64).T
    res = {"workload": f"X[{OCC_M},{OCC_K}] Student-t(3), 1% channels x100; W[{OCC_N},{OCC_K}]; NVFP4; h={h}; bf16 Y"}
    cases = {"plain": lambda: fp4.fp4_gemm(xq, wq, out=Y),
             "order2": lambda: fp4.fp4_hcp_gemm(X, W, xq, wq, hot, h, fp4.FP4_HCP_SINGLE, 2, out=Y, workspace=ws),
             "zeroed": lambda: fp4.fp4_hcp_gemm(X, W, x0q, wq, hot, h, fp4.FP4_HCP_SINGLE, 0, out=Y, workspace=ws),
             "order2_bf16_two_kernel": lambda: fp4.fp4_hcp_gemm(X, W, xq, wq, hot, h, fp4.FP4_HCP_TWO, 2, out=Y,
                                                                workspace=ws),
             "order2_fp8_two_kernel": lambda: fp4.fp4_hcp_gemm(X, W, xq, wq, hot, h, fp4.FP4_HCP_TWO_FP8, 2, out=Y,
                                                               workspace=ws),
             "zeroed_fp8_two_kernel": lambda: fp4.fp4_hcp_gemm(X, W, x0q, wq, hot, h, fp4.FP4_HCP_TWO_FP8, 0, out=Y,
                                                               workspace=ws)}
    for name, fn in cases.items():
        r = _rate("tensor", flops, _time_op(fn, flush, launches), pk)
        fn()
        got = Y.float().cpu().numpy()[rows].astype(np.float64)
        r["rel_err_pct"] = 100.0 * float(np.sqrt(((got - exact) ** 2).sum() / (exact ** 2).sum()))
        res[name] = r
    res["zeroed_quantize"] = _rate("hbm", OCC_M * OCC_K * (2 + 0.5 + 1 / 16), _time_op(
        lambda: fp4.fp4_hcp_quantize_zeroed(X, p, hot, h, out=x0q), flush, launches), pk)
    return res


def block_sweep(fp4, step, dev, flush, launches, pk):
    """Block sizes 16-128 with E4M3 (NVFP4-style) and E8M0 (MXFP4-style) scales on the step's X
    ("深度学习中的梯度计算基础" §4.2, §5.1): quantize throughput and the relative L2 error of the
    dequantized (STE forward) and the sigmoid-smoothed (beta 10, 40) reconstructions, in percent."""
    X = step.X
    n = X.numel()
    out = {"tensor": f"X[{M},{K}] ~N(0,1) bf16, RTN, row-major scales", "rows": []}
    for fmt, name in ((fp4.FP4_FMT_NVFP4, "E4M3"), (fp4.FP4_FMT_MXFP4, "E8M0")):
        for block in (16, 32, 64, 128):
            p = fp4.quant_params(fmt, sf_layout=fp4.FP4_SF_ROWMAJOR, block=block)
            q = fp4.alloc_qtensor(M, K, fmt, fp4.FP4_SF_ROWMAJOR, dev, block)
            t = _time_op(lambda: fp4.fp4_quantize(X, p, out=q), flush, launches)
            row = {"scale": name, "block": block, **_rate("hbm", n * (2 + 0.5 + 1.0 / block), t, pk)}
            for label, beta in (("ste", 0.0), ("soft_beta10", 10.0), ("soft_beta40", 40.0)):
                st = fp4.error_stats_from_sums(fp4.fp4_quant_error_sums(X, q, beta=beta).cpu(), n)
                row[f"rel_err_pct_{label}"] = 100.0 * st["rel_err"]
            out["rows"].append(row)
    return out


# Outlier clamping and compensation (the MSR write-up §三) on the hot-channel
# activations: X[16384,4096] Student-t(3) with 1% of the channels x100,
# W[4096,4096] ~N(0,0.02), NVFP4, q = 0.99, 64 dense compensation columns.
OCC_M, OCC_K, OCC_N, OCC_DENSE = 16384, 4096, 4096, 64


def time_occ(fp4, dev, flush, launches, pk):
    from fp4_block_scaled_e8m0_gb300 import inputs
    d = inputs.hcp_square(OCC_M, OCC_K, OCC_N)
    X, W = d["X"].to(dev), d["W"].to(dev)
    NV = fp4.FP4_FMT_NVFP4
    p = fp4.quant_params(NV)
    ws_t = torch.empty((fp4.load_library().fp4_occ_threshold_workspace_bytes(fp4.FP4_DTYPE_BF16),),
                       dtype=torch.uint8, device=dev)
    tau, n_out = fp4.fp4_occ_threshold(X, workspace=ws_t)
    counts = torch.empty((OCC_K,), dtype=torch.float32, device=dev)
    xq = fp4.alloc_qtensor(OCC_M, OCC_K, NV, fp4.FP4_SF_MMA, dev)
    fp4.fp4_occ_quantize(X, p, tau, out=xq, col_counts=counts)
    wq = fp4.fp4_quantize(W, p)
    xq_direct = fp4.fp4_quantize(X, p)
    cap = fp4.fp4_occ_max_outliers(OCC_M, OCC_K)
    ws = torch.empty((fp4.load_library().fp4_occ_gemm_workspace_bytes(OCC_M, OCC_N, OCC_K, OCC_DENSE, cap),),
                     dtype=torch.uint8, device=dev)
    Y = torch.empty((OCC_M, OCC_N), dtype=torch.bfloat16, device=dev)
    flops = 2 * OCC_M * OCC_N * OCC_K
    res = {"workload": f"X[{OCC_M},{OCC_K}] Student-t(3), 1% channels x100; W[{OCC_N},{OCC_K}]; NVFP4; q=0.99; "
                       f"{OCC_DENSE} dense columns; bf16 Y",
           "outliers": int(n_out.item()), "tau": float(tau.item())}
    res["threshold"] = _rate("hbm", OCC_M * OCC_K * 2, _time_op(
        lambda: fp4.fp4_occ_threshold(X, workspace=ws_t), flush, launches), pk)
    res["clamp_quantize"] = _rate("hbm", OCC_M * OCC_K * (2 + 0.5 + 1 / 16), _time_op(
        lambda: fp4.fp4_occ_quantize(X, p, tau, out=xq, col_counts=counts), flush, launches), pk)
    res["occ_gemm"] = _rate("tensor", flops, _time_op(
        lambda: fp4.fp4_occ_gemm(X, W, xq, wq, tau, counts, OCC_DENSE, cap, out=Y, workspace=ws), flush, launches), pk)
    res["plain_gemm"] = _rate("tensor", flops, _time_op(lambda: fp4.fp4_gemm(xq, wq, out=Y), flush, launches), pk)
    n = OCC_M * OCC_K
    res["quality_direct"] = fp4.error_stats_from_sums(fp4.fp4_quant_error_sums(X, xq_direct).cpu(), n)
    res["quality_occ"] = fp4.error_stats_from_sums(fp4.fp4_quant_error_sums(X, xq, tau).cpu(), n)
    return res


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        loaded = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in loaded if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for name, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(loaded)}


# ---------------------------------------------------------------------------
# roofline denominators
# ---------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp4_block_scaled_e8m0_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_traffic(op: str):
    """DRAM bytes per launch of `op` from the committed ncu summary, or None when
    the kernels changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("source_digest") != source_digest():
        return None
    v = d.get("ops", {}).get(op)
    return None if v is None else float(v)


# ---------------------------------------------------------------------------
# CPU legs (the oracle)
# ---------------------------------------------------------------------------
def oracle_step(Ms, Ns, Kk=K, seed=0):
    """The step's arithmetic on an Ms x Kk / Ns x Kk / Ms x Ns sample, by the oracle."""
    import oracle as o
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((Ms, Kk)).astype(np.float32)
    W = (rng.standard_normal((Ns, Kk)) * 0.02).astype(np.float32)
    dY = (rng.standard_normal((Ms, Ns)) * 1e-3).astype(np.float32)
    t0 = time.perf_counter()
    xq = o.quantize(X, o.NVFP4)
    wq = o.quantize(W, o.NVFP4)
    o.gemm(*xq[:2], *wq[:2], o.NVFP4, xq[2], wq[2])
    dyn = o.quantize(dY, o.NVFP4, "sr", rht=True, sr_seed=2, sr_stream=0, rht_seed=2)
    dym = o.quantize(dY, o.NVFP4, "sr", transpose=True, rht=True, sr_seed=2, sr_stream=2, rht_seed=2)
    wt = o.quantize(W, o.NVFP4, "sr", "2d", True, True, sr_seed=2, sr_stream=1, rht_seed=2)
    xt = o.quantize(X, o.NVFP4, "sr", transpose=True, rht=True, sr_seed=2, sr_stream=3, rht_seed=2)
    o.gemm(*dyn[:2], *wt[:2], o.NVFP4, dyn[2], wt[2])
    dw, _ = o.gemm(*dym[:2], *xt[:2], o.NVFP4, dym[2], xt[2])
    o.dge_backward(W, wq[1], o.NVFP4, wq[2], dw)
    return time.perf_counter() - t0


def cpu_cores() -> int:
    return os.cpu_count() or 1


def cpu_baseline(sample: str):
    Ms, Ns = (int(v) for v in sample.split("x"))
    t = oracle_step(Ms, Ns)
    flops = 3 * 2 * Ms * Ns * K
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"the full step on X[{Ms},{K}] W[{Ns},{K}] dY[{Ms},{Ns}] (numpy oracle; BLAS matmul may use all "
                      f"cores, elementwise steps one core); {t:.2f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    # each step: the oracle on a bounded sample, sized so that the run ends in minutes
    Ms, Ns = 16, 16
    for _ in range(args.warmup):
        oracle_step(Ms, Ns)
    ts = [oracle_step(Ms, Ns, seed=i) for i in range(args.steps)]
    t = float(np.mean(ts))
    flops = 3 * 2 * Ms * Ns * K
    value = flops / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64 (numpy oracle)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": f"M={Ms} N={Ns} K={K} per step"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"the full step on X[{Ms},{K}] W[{Ns},{K}] dY[{Ms},{Ns}] per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# multi-rank aggregation (replicas: each rank runs the whole step on its own
# data; the job's step time is the slowest rank's)
# ---------------------------------------------------------------------------
def reduce_step_time(t_local: float, dist, device) -> float:
    if dist is None:
        return t_local
    t = torch.tensor([t_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, t_step: float) -> float:
    """Whole-job TFLOP/s: every rank processes one step's GEMM flops per t_step."""
    return world * STEP_FLOPS / t_step / 1e12


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import fp4_block_scaled_e8m0_gb300 as fp4
    from fp4_block_scaled_e8m0_gb300 import build as fbuild
    from fp4_block_scaled_e8m0_gb300 import inputs
    if not os.path.exists(fbuild.lib_path()):
        if rank == 0:
            fbuild.build()
        if dist:
            dist.barrier()
    fp4.load_library()

    data = inputs.llama1b_mlp_up()
    host = {k: data[k].pin_memory() for k in ("X", "W", "dY")}
    X, W, dY = (host[k].to(dev) for k in ("X", "W", "dY"))
    step = Step(fp4, X, W, dY, dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    side = torch.cuda.Stream(device=dev)
    for i in range(args.warmup):
        step.run(i, side=side)
    torch.cuda.synchronize()
    if args.ext_only:
        if args.warmup < 1:
            step.run(0)
        ext = time_extensions(fp4, step, dev, flush, max(args.ext_launches, 1), peaks())
        if rank == 0:
            print(json.dumps({"extensions": ext}), flush=True)
        return

    names = list(OPS)
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    n_breakdown = min(args.steps, 20)
    ev_ops = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for n in names}
              for _ in range(n_breakdown)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)                    # L2 flush, outside the step's events
        ev_step[i][0].record(stream)
        step.run(args.warmup + i, side=side)
        ev_step[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    clk = clocks.stop()
    # per-op breakdown: further steps, each op alone on the stream with events
    # around it (outside the timed region, so the event records do not enter the
    # step time)
    for i in range(n_breakdown):
        flush.fill_(i & 0xFF)
        step.run(args.warmup + args.steps + i, ev_ops[i])
    torch.cuda.synchronize()
    step_s = np.array([a.elapsed_time(b) * 1e-3 for a, b in ev_step])
    op_s = {n: float(np.mean([e[n][0].elapsed_time(e[n][1]) * 1e-3 for e in ev_ops])) for n in names}
    t_step = reduce_step_time(float(step_s.mean()), dist, dev)
    status = fp4.fp4_sync_status() | fp4.fp4_sync_status(step.side_ctx)

    # ---- end to end through the C ABI with host buffers --------------------------
    h_out = {"Y": torch.empty((M, N), dtype=torch.bfloat16).pin_memory(),
             "dX": torch.empty((M, K), dtype=torch.bfloat16).pin_memory(),
             "dW": torch.empty((N, K), dtype=torch.float32).pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    # Copies run on their own streams and overlap with the computation: each
    # input is waited for just before the first op that reads it, and each
    # result is copied back as soon as the op that produces it has finished.
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e = []
    for i in range(args.e2e_steps):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        arrived = {k: torch.cuda.Event() for k in ("X", "W", "dY")}
        s_h2d.wait_stream(stream)
        with torch.cuda.stream(s_h2d):
            for k, t in (("X", X), ("W", W), ("dY", dY)):   # in the order the step needs them
                t.copy_(host[k], non_blocking=True)
                arrived[k].record(s_h2d)

        def copy_back(name, src, s):
            done = torch.cuda.Event()
            done.record(s)
            s_d2h.wait_event(done)
            with torch.cuda.stream(s_d2h):
                h_out[name].copy_(src, non_blocking=True)

        step.run(10_000 + i,
                 before={"quant_x_dual": lambda s: s.wait_event(arrived["X"]),
                         "quant_w_dual": lambda s: s.wait_event(arrived["W"]),
                         "quant_dy_dual": lambda s: s.wait_event(arrived["dY"])},
                 after={"fprop": lambda s: copy_back("Y", step.Y, s),
                        "dgrad": lambda s: copy_back("dX", step.dX, s),
                        "dge": lambda s: copy_back("dW", step.dWd, s)},
                 side=side)
        stream.wait_stream(s_d2h)
        b.record(stream)
        b.synchronize()
        e2e.append(a.elapsed_time(b) * 1e-3)
    t_e2e = float(np.mean(e2e)) if e2e else float("nan")

    pk = peaks()
    extensions = time_extensions(fp4, step, dev, flush, args.ext_launches, pk) if args.ext_launches > 0 else {}

    # ---- roofline of the dominant kernel --------------------------------------------
    dom = max(names, key=lambda n: op_s[n])
    kind, units = OPS[dom]
    if kind == "tensor":
        peak = pk["bf16_tflops_sustained"] * FP4_OVER_BF16
        achieved = units / op_s[dom] / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{pk['source']} bf16 sustained x {FP4_OVER_BF16:g} (nominal FP4:BF16)"}
    else:
        peak = pk["hbm_gbs"]
        achieved = units / op_s[dom] / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{pk['source']} HBM copy"}
    roof["kernel"] = dom
    traffic = measured_traffic(dom)
    roof["traffic"] = traffic

    breakdown = {}
    for n in names:
        k_, u = OPS[n]
        rate = u / op_s[n] / (1e12 if k_ == "tensor" else 1e9)
        pkv = pk["bf16_tflops_sustained"] * FP4_OVER_BF16 if k_ == "tensor" else pk["hbm_gbs"]
        breakdown[n] = {"us": op_s[n] * 1e6, "rate": rate, "unit": "TFLOP/s" if k_ == "tensor" else "GB/s",
                        "frac": rate / pkv}
    q_names = [n for n in names if OPS[n][0] == "hbm" and n.startswith("quant")]
    q_bytes = sum(OPS[n][1] for n in q_names)
    q_time = sum(op_s[n] for n in q_names)
    g_time = sum(op_s[n] for n in names if OPS[n][0] == "tensor")

    value = job_value(world, t_step)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3 block scale x fp32 tensor scale), fp32 accumulate",
        "data": "synthetic (seeded numpy: X~N(0,1), W~N(0,0.02), dY~N(0,1e-3))",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "parallelism": "replicas" if world > 1 else "1 gpu",
                   "l2": "flushed before each timed step (512 MiB write)"},
        "quantize_gbs": q_bytes / q_time / 1e9, "gemm_tflops": 3 * GEMM_FLOPS / g_time / 1e12,
        "step_roofline_frac": (sum(OPS[n][1] / (pk['bf16_tflops_sustained'] * FP4_OVER_BF16 * 1e12)
                                   if OPS[n][0] == "tensor" else OPS[n][1] / (pk['hbm_gbs'] * 1e9) for n in names)
                               / t_step),
        "ops": breakdown, "roofline": roof, "clocks": clk,
        "e2e": {"value": world * STEP_FLOPS / t_e2e / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3},
        "extensions": extensions,
        "gpu_launches": sum(KERNELS_PER_OP.values()) * args.steps, "wall_s_timed_region": wall,
        "device_status": status,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_sample)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
