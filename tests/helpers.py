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


# Guard bands around outputs (a stand-in for a memory checker, which is not
# available on the GPU pool): sentinel bit patterns -- NaNs with a payload no
# kernel computes -- fill the rows above and below an output and the columns
# right of it up to its row stride; after the call every sentinel must be
# unchanged.  Tiled kernels go wrong at their edges ("GEMM o Coração
# Matemático", §4.2), e.g. a staged TMA store built with a wrong extent.
_SENTINEL = {torch.bfloat16: (torch.int16, 0x7FA5), torch.float16: (torch.int16, 0x7E5A),
             torch.float32: (torch.int32, 0x7FA5A5A5)}
GUARD_ROWS_ABOVE = 4
GUARD_ROWS_BELOW = 130          # more than one 128-row tile
GUARD_COLS_BYTES = 128          # one TMA store box


class Guarded:
    """A rows x cols output inside a larger device allocation of sentinels.

    ``view`` is the output (row stride ``ld``) to pass to the library; it
    holds ``init`` (a rows x cols tensor) or, without one, the value ``fill``.
    ``ld`` defaults to cols + 128 bytes of guard columns, rounded to 16 bytes;
    pass ``ld=cols`` where the callee fixes the row stride (then only the rows
    above and below guard it).  ``check()`` asserts every sentinel unchanged;
    ``cpu()`` checks and returns the output."""

    def __init__(self, rows, cols, dtype, init=None, fill=None, ld=None,
                 above=GUARD_ROWS_ABOVE, below=GUARD_ROWS_BELOW, device="cuda"):
        ity, bits = _SENTINEL[dtype]
        esz = torch.empty((), dtype=dtype).element_size()
        if ld is None:
            ld = round_up(cols + GUARD_COLS_BYTES // esz, 16 // esz)
        assert ld >= cols and (ld * esz) % 16 == 0, (ld, cols, esz)
        self.rows, self.cols, self.ld, self.above, self.below = rows, cols, ld, above, below
        self.dtype, self.ity, self.bits = dtype, ity, bits
        self.full = torch.full((above + rows + below, ld), bits, dtype=ity,
                               device=device).view(dtype)
        self.view = self.full[above:above + rows, :cols]
        if init is not None:
            self.view.copy_(init)
        elif fill is not None:
            self.view.fill_(fill)
        # the library may be called on another stream than the one that
        # filled the buffer
        torch.cuda.current_stream(self.full.device).synchronize()

    def check(self, what: str = "") -> None:
        full = self.full.view(self.ity).cpu()
        a, r = self.above, self.rows
        regions = [("rows above", full[:a]), ("rows below", full[a + r:]),
                   ("columns right", full[a:a + r, self.cols:])]
        for name, reg in regions:
            bad = reg != self.bits
            if bool(bad.any()):
                idx = bad.nonzero()[:5].tolist()
                raise AssertionError(f"{what}: {int(bad.sum())} guard elements ({name}) "
                                     f"overwritten, e.g. {idx}")

    def cpu(self, what: str = "") -> torch.Tensor:
        self.check(what)
        return self.view.cpu()


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
