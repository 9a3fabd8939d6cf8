"""Oracle evaluation of many query tokens in parallel worker processes (test infrastructure).

The workers import only numpy and the oracle (no torch, no CUDA), and the pool is started with
the "spawn" method so that no worker inherits a CUDA context from the test process."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from oracle import attention, codec, pack


def _one_unit(args):
    q_bits, lat_bits, rope_bits, scale = args
    rows = pack.encode_rows(lat_bits, rope_bits)
    c = attention.dequant_rows(rows)
    return attention.attend(codec.bf16_bits_to_f64(q_bits), c, scale)


def attend_units(jobs, workers: int | None = None):
    """jobs: list of (q_bits uint16 [H, 576], latent bits [n, 512], rope bits [n, 64], scale).
    Returns a list of (out float64 [H, 512], lse float64 [H]) in job order."""
    if not jobs:
        return []
    n = workers or max(1, min(8, (os.cpu_count() or 1)))
    if n == 1 or len(jobs) == 1:
        return [_one_unit(j) for j in jobs]
    with mp.get_context("spawn").Pool(n) as pool:
        return pool.map(_one_unit, jobs, chunksize=max(1, len(jobs) // (4 * n)))
