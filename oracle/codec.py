"""Value codecs: bf16, FP8-E4M3 and FP4-e2m1 (oracle; test infrastructure only).

Format facts, from "Prime Inference" (translated page), section "Making room
for low-latency decode", and "Prime Inference: serving GLM-5.3 to agents is a
KV-cache problem", section "Four bits per latent value": latent values are
stored in four bits (NVFP4, i.e. the e2m1 element type) with one FP8 scale per
16 values, and the rope part is stored as FP8. The FP8 type is E4M3 (the
NVFP4 block-scale type; the same E4M3 is used for the rope bytes).

E4M3 ("fn" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent
field 0 is subnormal (m/8 * 2^-6); 0x7F/0xFF are NaN; largest finite 448.
e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
{0, 0.5, 1, 1.5, 2, 3, 4, 6} for codes 0..7, bit 3 is the sign.

Rounding (the pages do not state it; the reading taken is IEEE-style):
round to nearest, ties to the even code, saturating at the largest finite
magnitude; the sign of the input is kept, including -0.0 and values that
round to zero.
"""
from __future__ import annotations

import numpy as np

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E4M3_MAX = 448.0


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """Value of E4M3 bytes as float64 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = s * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


# All non-negative finite E4M3 magnitudes, in code order 0x00..0x7E (increasing).
E4M3_GRID = e4m3_decode(np.arange(0x7F))


def _nearest_even(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid value nearest to mag (grid increasing, mag >= 0).

    Ties go to the even index; magnitudes above the last grid value saturate
    to it. The distance comparison is done on float64 values; the callers only
    pass magnitudes whose distance to a midpoint is either exactly zero or far
    larger than float64 rounding (see quantise_block).
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(grid, mag, side="left")          # first grid >= mag
    hi = np.clip(hi, 0, grid.size - 1)
    lo = np.clip(hi - 1, 0, grid.size - 1)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= grid[-1], grid.size - 1, idx)
    return idx.astype(np.int64)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round float64 values to E4M3 bytes: nearest, ties to even, saturating.

    Non-finite inputs (a reading; the pages say nothing about them): +-inf
    saturates to +-448 like any value past the largest finite magnitude, and
    NaN becomes the E4M3 NaN pattern 0x7F with the input's sign bit kept
    (0x7F or 0xFF).
    """
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    idx = _nearest_even(np.where(nan, 0.0, np.abs(x)), E4M3_GRID)
    idx = np.where(nan, 0x7F, idx)
    sign = np.signbit(x).astype(np.int64) << 7
    return (idx | sign).astype(np.uint8)


def e2m1_decode(code: np.ndarray) -> np.ndarray:
    """Value of 4-bit e2m1 codes (0..15) as float64."""
    c = np.asarray(code, dtype=np.int64)
    return np.where(c & 0x8, -1.0, 1.0) * E2M1_GRID[c & 0x7]


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round float64 values to e2m1 codes (0..15): nearest, ties to even, saturating at 6.

    e2m1 has no NaN or infinity. Reading for non-finite inputs: +-inf
    saturates to +-6 (code 7 with the sign bit), and NaN gets magnitude code 0
    with its sign bit kept.
    """
    v = np.asarray(v, dtype=np.float64)
    idx = _nearest_even(np.where(np.isnan(v), 0.0, np.abs(v)), E2M1_GRID)
    sign = np.signbit(v).astype(np.int64) << 3
    return (idx | sign).astype(np.uint8)
