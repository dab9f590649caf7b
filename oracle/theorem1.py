"""Theorem 1 diagnostic -- TEST INFRASTRUCTURE ONLY.  Parity unpinned.

"MXNorm: Reusing MXFP block scales for efficient tensor normalisation",
Resumen tecnico, 2. Metodologia, "Fundamentos Teoricos": the power mean of a
row's block scales follows the row's RMS up to a constant c(p, B), which the
pages call precomputed but never print.  The library runs with c = 1, so
for each row the product

    ratio = RMS_exact(x) * inv_rms,   RMS_exact = sqrt(mean_j x_j^2)

is that constant's empirical value for the row.  This module computes its
distribution on the synthetic workloads through the oracle; the pages give
no number to compare it with, so nothing here is pinned to the pages.

What the E8M0 rule itself fixes, whatever the data (the bounds the tests
check): a block whose maximum magnitude a is above the E8M0 clamp gets the
scale s = 2^(floor(log2 a) - emax), so 2^emax s <= a < 2^(emax+1) s, and its
32 values have a sum of squares in [a^2, 32 a^2].  Summed over the K = H/32
blocks of a row with no zero block:

    p = 2:  2^emax / sqrt(32) <= RMS / M_2 < 2^(emax+1)
    p = 1:  2^emax / sqrt(32) <= RMS / M_1 < 2^(emax+1) sqrt(K)

(M_1 <= M_2 <= sqrt(K) M_1).  A constant row of value v gives exactly
|v| / 2^(floor(log2 |v|) - emax), in [2^emax, 2^(emax+1)).

For the rotated formats the scales belong to the rotated row, whose RMS is
x's (H16 / 4 and H32 / sqrt(32) are orthonormal) up to the fp32 rounding of
the rotation.

tests/golden/print_theorem1_table.py prints the distribution per workload
as a Markdown table with summary().
"""
from __future__ import annotations

import numpy as np

from . import mxnorm_quant

EMAX = {"mxfp8": 8, "mxfp8_h16": 8, "mxfp8_h32": 8, "mxfp4": 2, "mxfp4_h16": 2, "mxfp4_h32": 2}


def rms_exact(x_bits: np.ndarray) -> np.ndarray:
    """Per-row RMS of bf16 rows, in fp64 (bf16 -> fp64 is exact)."""
    b = np.ascontiguousarray(x_bits, dtype=np.uint16)
    v = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.sqrt(np.mean(v * v, axis=1))


def ratio(x_bits: np.ndarray, p: int, fmt: str) -> np.ndarray:
    """RMS_exact(row) * inv_rms(row) from the oracle's estimate (c = 1)."""
    _, _, inv = mxnorm_quant(x_bits, p, fmt)
    return rms_exact(x_bits) * inv.astype(np.float64)


def bounds(p: int, fmt: str, H: int):
    """[lo, hi) that the E8M0 rule forces on ratio() for rows with no zero
    block (and no block below the E8M0 clamp)."""
    emax = EMAX[fmt]
    lo = 2.0 ** emax / np.sqrt(32.0)
    hi = 2.0 ** (emax + 1) * (1.0 if p == 2 else np.sqrt(H / 32))
    return lo, hi


def summary(x_bits: np.ndarray, p: int, fmt: str) -> dict:
    r = ratio(x_bits, p, fmt)
    return {"mean": float(r.mean()), "std": float(r.std()), "min": float(r.min()), "max": float(r.max()),
            "cv": float(r.std() / r.mean()), "rows": int(r.size)}
