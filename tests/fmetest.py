"""Helpers shared by the tests: reading the library's tiled scale layout back into
logical [rows x C] matrices (an independent restatement of the layout in
include/fme.h), moving tensors between torch and numpy, and the GEMM tolerance."""
from __future__ import annotations

import numpy as np


def group_tiles(offsets: np.ndarray) -> np.ndarray:
    """128-row tile prefix: tiles[g] = sum_{g'<g} ceil(n_g'/128)."""
    counts = np.diff(np.asarray(offsets, np.int64))
    return np.concatenate([[0], np.cumsum((counts + 127) // 128)]).astype(np.int64)


def padded_rows(offsets: np.ndarray) -> np.ndarray:
    """Padded row of every logical row under per-group 128-row padding."""
    off = np.asarray(offsets, np.int64)
    tiles = group_tiles(off)
    rows = int(off[-1])
    g = np.searchsorted(off, np.arange(rows), side="right") - 1
    return 128 * tiles[g] + (np.arange(rows) - off[g])


def sf_index(pr: np.ndarray, c: np.ndarray, c_logical: int) -> np.ndarray:
    c4 = (c_logical + 3) // 4 * 4
    return ((pr // 128) * (c4 // 4) + c // 4) * 512 + (pr % 32) * 16 + ((pr % 128) // 32) * 4 + c % 4


def unswizzle(sf_flat: np.ndarray, rows: int, c_logical: int, offsets=None) -> np.ndarray:
    """Tiled scale bytes -> logical [rows x c_logical] matrix."""
    if offsets is None:
        offsets = np.array([0, rows])
    pr = padded_rows(offsets)
    assert len(pr) == rows
    c = np.arange(c_logical)
    idx = sf_index(pr[:, None], c[None, :], c_logical)
    return np.asarray(sf_flat)[idx]


def to_np(t) -> np.ndarray:
    return t.detach().cpu().numpy()


from fp8_moe_expert_gb300.synth import bf16_bits_np  # noqa: E402,F401  (re-exported for the tests)


def bf16_tensor(bits: np.ndarray, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_f64(t) -> np.ndarray:
    import torch

    return t.detach().to(torch.float64).cpu().numpy()


def check_gemm_tolerance(y: np.ndarray, y_ref: np.ndarray, rms: float | None = None, what: str = ""):
    """|y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref), element by element."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    if rms is None:
        rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    err = np.abs(y - y_ref)
    bound = 8e-3 * np.abs(y_ref) + 1e-3 * rms
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: got {y[tuple(i)]:.6g} want {y_ref[tuple(i)]:.6g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; {detail}")
    return float((err / (np.abs(y_ref) + rms + 1e-30)).max()) if y.size else 0.0
