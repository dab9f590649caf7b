"""Seeded synthetic activations shaped like Llama-3 hidden states.

This module holds no MXNorm arithmetic: it only draws random numbers and
rounds them to bf16.  Both the CUDA path and the CPU oracle consume its
output, so it imports neither.

The MXNorm pages validate on Llama 3 125M / 1B / 8B pre-training
("MXNorm: Reusing MXFP block scales ...", Resumen tecnico, section 4, and
the English abstract) and the MXFP4 page on Llama 3.1-8B with outlier-heavy
activations ("Entrenamiento Previo ... con MXFP4", Enunciado del Problema).
No activations ship with the pages, so heavy-tailed stand-ins are drawn:

  * "normal":       x = N(0, 1), with a fixed list of outlier channels scaled.
  * "t4_lognormal": x[t, j] = t4[t, j] * g[j] * o[j], where t4 is Student-t
                    with 4 degrees of freedom drawn as Z / sqrt(G / 2) with
                    Z ~ N(0, 1) and G ~ Gamma(shape 2, scale 1) (so 2G is
                    chi-square with 4 dof), g[j] = exp(0.5 * N(0, 1)) is a
                    per-channel lognormal gain shared by all rows, and o[j]
                    is the outlier gain on round(frac * H) channels picked by
                    a seeded permutation (1 elsewhere).

All draws come from numpy's PCG64 in float32, in a fixed order: channel
gains, outlier channels, then the rows in chunks of CHUNK_ROWS (Z then G per
chunk).  Values are rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

CHUNK_ROWS = 1024


@dataclass(frozen=True)
class Workload:
    """One seeded synthetic activation workload: T rows of H bf16 values
    drawn from `dist` with per-channel gains and `outlier_frac` of the
    channels (or the listed `outlier_channels`) scaled by `outlier_gain`."""
    name: str
    T: int
    H: int
    seed: int
    dist: str
    fmt: str
    ps: tuple
    outlier_gain: float
    outlier_frac: float = 0.0
    outlier_channels: tuple = field(default_factory=tuple)
    note: str = ""

    @property
    def K(self) -> int:
        """MX blocks per row."""
        return self.H // 32


WORKLOADS = {
    "tiny_64x256": Workload(
        "tiny_64x256", 64, 256, 0, "normal", "mxfp8", (2,), 50.0,
        outlier_channels=(17, 200), note="tiny oracle case, N(0,1), channels 17 and 200 x50"),
    "llama3_125m_16384x768": Workload(
        "llama3_125m_16384x768", 16384, 768, 1, "t4_lognormal", "mxfp8", (1, 2), 30.0,
        outlier_frac=0.01, note="Llama-3-125M-shaped, 8 seqs x 2048 tokens"),
    "llama3_1b_32768x2048": Workload(
        "llama3_1b_32768x2048", 32768, 2048, 2, "t4_lognormal", "mxfp8", (2,), 30.0,
        outlier_frac=0.005, note="Llama-3-1B-shaped, 16 x 2048 tokens"),
    "llama3_8b_65536x4096": Workload(
        "llama3_8b_65536x4096", 65536, 4096, 3, "t4_lognormal", "mxfp8", (1, 2), 100.0,
        outlier_frac=0.001, note="Llama-3-8B-shaped, 16 x 4096 tokens"),
    "llama3_8b_mxfp4_h16_65536x4096": Workload(
        "llama3_8b_mxfp4_h16_65536x4096", 65536, 4096, 4, "t4_lognormal", "mxfp4_h16", (2,), 100.0,
        outlier_frac=0.001, note="Llama-3-8B-shaped, H16 rotation then MXFP4 E2M1"),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values (finite, far from overflow) to bf16 bit patterns,
    nearest with ties to even, by integer arithmetic on the float32 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> their float32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def channel_gains(w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Per-channel gains shared by every row of w: exp(0.5 Z) times the
    outlier gain on the outlier channels (a seeded permutation), or ones
    with the listed outlier channels for the normal workload."""
    H = w.H
    if w.dist == "normal":
        g = np.ones(H, np.float32)
        g[list(w.outlier_channels)] = np.float32(w.outlier_gain)
        return g
    g = np.exp(np.float32(0.5) * rng.standard_normal(H, dtype=np.float32)).astype(np.float32)
    n_out = int(round(w.outlier_frac * H))
    chans = rng.permutation(H)[:n_out]
    g[chans] *= np.float32(w.outlier_gain)
    return g


def outlier_channels(w: Workload) -> np.ndarray:
    """The outlier channel indices the generator picks for w (sorted)."""
    if w.dist == "normal":
        return np.array(sorted(w.outlier_channels))
    rng = np.random.Generator(np.random.PCG64(w.seed))
    rng.standard_normal(w.H, dtype=np.float32)
    return np.sort(rng.permutation(w.H)[: int(round(w.outlier_frac * w.H))])


def make_activations(w: Workload, rows: int | None = None) -> np.ndarray:
    """bf16 bit patterns [rows, H] (rows defaults to w.T); the first `rows`
    rows of the full workload, identical whatever `rows` is."""
    T = w.T if rows is None else int(rows)
    rng = np.random.Generator(np.random.PCG64(w.seed))
    g = channel_gains(w, rng)
    out = np.empty((T, w.H), np.uint16)
    for r0 in range(0, T, CHUNK_ROWS):
        n = min(CHUNK_ROWS, w.T - r0)
        z = rng.standard_normal((n, w.H), dtype=np.float32)
        if w.dist == "normal":
            x = z
        else:
            gam = rng.standard_gamma(np.float32(2.0), size=(n, w.H), dtype=np.float32)
            x = z / np.sqrt(gam * np.float32(0.5))
        x *= g
        take = min(n, T - r0)
        out[r0:r0 + take] = f32_to_bf16_bits(x[:take])
        if r0 + n >= T:
            break
    return out


def make_random_rows(T: int, H: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """Plain N(0, scale^2) bf16 rows for ragged / edge-case shapes."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32) * np.float32(scale))
