"""Oracle evaluation of many query tokens in parallel worker processes (test infrastructure).

The workers import only numpy and the oracle (no torch, no CUDA), and the pool is started with
the "spawn" method so that no worker inherits a CUDA context from the test process."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from oracle import attention, codec, fp8rows, pack


def _rows_values(lat_bits, rope_bits, fmt):
    """Dequantised selected rows of a unit in the cache format fmt: "nvfp4" (the 352-byte rows),
    "fp8" (576-byte FP8 rows packed from bf16), "staged" (FP8 copies of the NVFP4 rows) or "token"
    (672-byte per-token FP8 rows)."""
    if fmt == "nvfp4":
        return attention.dequant_rows(pack.encode_rows(lat_bits, rope_bits))
    if fmt == "fp8":
        return fp8rows.dequant_rows_fp8(fp8rows.encode_rows_fp8(lat_bits, rope_bits))
    if fmt == "staged":
        return fp8rows.dequant_rows_fp8(fp8rows.stage_rows(pack.encode_rows(lat_bits, rope_bits)))
    if fmt == "token":
        return fp8rows.dequant_rows_token(fp8rows.encode_rows_token(lat_bits, rope_bits))
    raise ValueError(fmt)


def _one_unit(args):
    q_bits, lat_bits, rope_bits, scale, fmt = args if len(args) == 5 else (*args, "nvfp4")
    c = _rows_values(lat_bits, rope_bits, fmt)
    return attention.attend(codec.bf16_bits_to_f64(q_bits), c, scale)


def attend_units(jobs, workers: int | None = None):
    """jobs: list of (q_bits uint16 [H, 576], latent bits [n, 512], rope bits [n, 64], scale[, fmt]).
    Returns a list of (out float64 [H, 512], lse float64 [H]) in job order."""
    if not jobs:
        return []
    n = workers or max(1, min(8, (os.cpu_count() or 1)))
    if n == 1 or len(jobs) == 1:
        return [_one_unit(j) for j in jobs]
    with mp.get_context("spawn").Pool(n) as pool:
        return pool.map(_one_unit, jobs, chunksize=max(1, len(jobs) // (4 * n)))
