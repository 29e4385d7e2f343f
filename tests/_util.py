"""Helpers shared by the tests (no method arithmetic: layout and comparison only)."""
import numpy as np
import torch


def untile_scales(buf: np.ndarray, rows: int, nsf: int) -> np.ndarray:
    """Scale bytes in the MMA layout (512-byte atoms of 128 rows x 4 scales,
    rows padded to 128, scales per row padded to a multiple of 4) -> [rows][nsf]."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    nsf_pad = buf.size // (((rows + 127) // 128) * 128)
    r = np.arange(rows).reshape(-1, 1)
    j = np.arange(nsf).reshape(1, -1)
    off = ((r // 128) * (nsf_pad // 4) + j // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (j % 4)
    return buf[off]


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def mismatch_report(got, want, label, limit=8):
    got = np.asarray(got)
    want = np.asarray(want)
    bad = np.argwhere(got != want)
    lines = [f"{label}: {len(bad)} mismatches of {want.size}"]
    for idx in bad[:limit]:
        idx = tuple(idx)
        lines.append(f"  at {idx}: got {got[idx]!r} want {want[idx]!r}")
    return "\n".join(lines)
