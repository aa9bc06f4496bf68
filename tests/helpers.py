"""Shared helpers for the parity tests: padded storage, tolerance checks.

Tolerances (the acceptance bar of this library):
* bf16 / fp16 outputs: |y - yhat| <= 1e-2 + 1e-2 |yhat| element-wise (the
  atol + rtol form of "为什么 GEMM 是 CUDA 的必修课", 精度 section);
* fp32 outputs: |y - yhat| <= 1e-4 sqrt(K) max|yhat|;
* every output finite.
"""
from __future__ import annotations

import math

import numpy as np
import torch

ATOL = 1e-2
RTOL = 1e-2


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def padded(t: torch.Tensor, ld: int, fill: float = 0.0) -> torch.Tensor:
    """rows x ld storage holding t in its first columns; the padding carries
    `fill` so a kernel that reads past the row shows it."""
    rows, cols = t.shape
    out = torch.full((rows, ld), fill, dtype=t.dtype)
    out[:, :cols] = t
    return out


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def check_half(y: np.ndarray, yhat: np.ndarray, what: str = "") -> dict:
    assert y.shape == yhat.shape, (y.shape, yhat.shape)
    assert np.isfinite(y).all(), f"{what}: non-finite outputs"
    err = np.abs(y - yhat)
    bound = ATOL + RTOL * np.abs(yhat)
    bad = err > bound
    stats = report(y, yhat)
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, e.g. {idx}; "
                             f"{stats}")
    return stats


def check_f32(y: np.ndarray, yhat: np.ndarray, K: int, what: str = "") -> dict:
    assert y.shape == yhat.shape
    assert np.isfinite(y).all(), f"{what}: non-finite outputs"
    scale = float(np.abs(yhat).max()) if yhat.size else 0.0
    bound = 1e-4 * math.sqrt(max(K, 1)) * scale
    err = float(np.abs(y - yhat).max()) if y.size else 0.0
    stats = report(y, yhat)
    assert err <= bound, f"{what}: max error {err} > {bound}; {stats}"
    return stats


def report(y: np.ndarray, yhat: np.ndarray) -> dict:
    if y.size == 0:
        return {"max_abs": 0.0, "max_rel": 0.0, "frac_rel_gt_1pct": 0.0}
    err = np.abs(y - yhat)
    rel = err / np.maximum(np.abs(yhat), 1e-30)
    return {"max_abs": float(err.max()), "max_rel": float(rel.max()),
            "frac_rel_gt_1pct": float((rel > 1e-2).mean())}


def check_two_stage(y, yhat, prop_bound, what=""):
    """Output of a composition whose intermediate is stored in bf16 (the full
    MLP: Y in bf16 between its two GEMMs).  The single-GEMM bound is widened by
    the propagated rounding of the intermediate, prop_bound = 2^-8 * |Y| |W|
    computed from the oracle's exact intermediate (2^-8 covers the bf16 store,
    2^-9, plus the FP32 arithmetic before it)."""
    assert y.shape == yhat.shape
    assert np.isfinite(y).all(), f"{what}: non-finite outputs"
    err = np.abs(y - yhat)
    bound = ATOL + RTOL * np.abs(yhat) + prop_bound
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, e.g. {idx}; "
                             f"{report(y, yhat)}")
    return report(y, yhat)
