"""Comparison rules between the GPU output and the FP64 oracle.

The order and the thresholds follow the "Xe2 ESIMD GEMM" page, section
"Correctness testing": look for NaN in the output first (a NaN would slip
through a ratio test), then require a relative RMS error below 0.5%.  On top
of that every element must satisfy |c - r| <= 1e-2 * (|r| + 1).

rel_rms is read as the norm ratio ||C - R||_2 / ||R||_2 over all compared
elements (the page does not define it; the mean of elementwise relative
errors would blow up near zero).
"""
from __future__ import annotations

import numpy as np

REL_RMS_MAX = 5e-3
ELEM_ABS = 1e-2


class ParityError(AssertionError):
    pass


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """GPU output (binary16 bit patterns) as float64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def check(c: np.ndarray, r: np.ndarray, what: str = "") -> dict:
    """Compare GPU values ``c`` with oracle values ``r`` (both float64).

    Raises ParityError on failure; returns the measured errors otherwise.
    """
    c = np.asarray(c, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if c.shape != r.shape:
        raise ParityError(f"{what}: shape {c.shape} vs oracle {r.shape}")
    bad = ~np.isfinite(c)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise ParityError(f"{what}: {int(bad.sum())} non-finite outputs, "
                          f"first at {tuple(idx)} = {c[tuple(idx)]}")
    diff = c - r
    rnorm = float(np.sqrt(np.sum(r * r)))
    dnorm = float(np.sqrt(np.sum(diff * diff)))
    rel_rms = dnorm / rnorm if rnorm > 0 else (0.0 if dnorm == 0 else np.inf)
    if not rel_rms < REL_RMS_MAX:
        raise ParityError(f"{what}: rel_rms {rel_rms:.3e} >= {REL_RMS_MAX}")
    lim = ELEM_ABS * (np.abs(r) + 1.0)
    over = np.abs(diff) > lim
    if over.any():
        idx = tuple(np.argwhere(over)[0])
        raise ParityError(f"{what}: {int(over.sum())} elements over the "
                          f"per-element bound, first at {idx}: gpu {c[idx]} "
                          f"oracle {r[idx]}")
    return {"rel_rms": rel_rms,
            "max_abs_err": float(np.abs(diff).max()) if diff.size else 0.0,
            "n": int(c.size)}
