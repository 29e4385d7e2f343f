"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random tensors; it holds none of the quantization
arithmetic.  Values come from numpy's PCG64 generator (identical on x86 and
Arm) in fp32 and are rounded to bf16 by torch.

Workloads (shapes stand in for the LLaMA-60M-to-13B models of the pages; no
dataset is involved):

* ``linear_fprop_small``  X 256x512 ~N(0,1), W 512x512 ~N(0,0.02); seed 0
* ``nvfp4_square``        T 4096x4096 ~N(0,1) with 64 random columns x100
                          (seed 1); dy ~N(0,1) (seed 101)
* ``llama1b_mlp_up``      X 8192x2048 ~N(0,1), W 5632x2048 ~N(0,0.02),
                          dY 8192x5632 ~N(0,1e-3); seed 2
* ``ffn7b``               X 16384x4096 Student-t(3) with 41 (1% of K) random
                          channels x100, W 11008x4096 ~N(0,0.02),
                          dY 16384x11008 ~N(0,1e-3); seed 3
* ``hcp_square``          X as ffn7b, W 4096x4096 ~N(0,0.02) (seed 4)
"""
from __future__ import annotations

import numpy as np
import torch


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def student_t(rng: np.random.Generator, shape, nu: float = 3.0) -> np.ndarray:
    return rng.standard_t(nu, size=shape).astype(np.float32)


def plant_hot_channels(rng: np.random.Generator, a: np.ndarray, count: int, factor: float = 100.0):
    """Scale ``count`` random columns by ``factor`` (persistent hot channels)."""
    cols = np.sort(rng.permutation(a.shape[1])[:count])
    a[:, cols] *= np.float32(factor)
    return cols


def linear_fprop_small():
    rng = _rng(0)
    return {"X": to_bf16(normal(rng, (256, 512))), "W": to_bf16(normal(rng, (512, 512), 0.02))}


def nvfp4_square(n: int = 4096):
    rng = _rng(1)
    t = normal(rng, (n, n))
    cols = plant_hot_channels(rng, t, 64 * n // 4096 or 1)
    dy = normal(_rng(101), (n, n))
    return {"T": to_bf16(t), "dy": to_bf16(dy), "hot_cols": cols}


def llama1b_mlp_up(m: int = 8192, k: int = 2048, n: int = 5632):
    rng = _rng(2)
    return {"X": to_bf16(normal(rng, (m, k))),
            "W": to_bf16(normal(rng, (n, k), 0.02)),
            "dY": to_bf16(normal(rng, (m, n), 1e-3))}


def _ffn_x(m: int, k: int):
    rng = _rng(3)
    x = student_t(rng, (m, k))
    cols = plant_hot_channels(rng, x, max(1, round(0.01 * k)))
    return rng, x, cols


def ffn7b(m: int = 16384, k: int = 4096, n: int = 11008, with_dy: bool = True):
    rng, x, cols = _ffn_x(m, k)
    out = {"X": to_bf16(x), "W": to_bf16(normal(rng, (n, k), 0.02)), "hot_cols": cols}
    if with_dy:
        out["dY"] = to_bf16(normal(rng, (m, n), 1e-3))
    return out


def hcp_square(m: int = 16384, k: int = 4096, n: int = 4096):
    _, x, cols = _ffn_x(m, k)
    w = normal(_rng(4), (n, k), 0.02)
    return {"X": to_bf16(x), "W": to_bf16(w), "hot_cols": cols}
