"""Timing the CPU oracle on query tokens of a decode workload (test and benchmark infrastructure).

Each query token (unit) is turned into a self-contained oracle call: the unit's selected rows are
drawn with the workload's own per-page row generator, encoded by the oracle's pack, and laid out
in a compact paged cache (32 pages of 64 rows for 2,048 entries) whose page table and index list
reach exactly those rows in the unit's order. attention.sparse_decode on that call does the same
work as on the full cache (validity, page lookup, gather, dequantisation, attention), without
holding the multi-GB cache in host memory.

Workers are started with the "spawn" method, import only numpy and this package, and keep the
prepared units in process memory, so a timed step moves only unit numbers and results.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import platform
import time

import numpy as np

from . import attention, pack

_UNITS = None      # per worker process: list of prepared units


_ARM_PARTS = {(0x41, 0xd4f): "Arm Neoverse V2", (0x41, 0xd40): "Arm Neoverse V1", (0x41, 0xd0c): "Arm Neoverse N1",
              (0x41, 0xd49): "Arm Neoverse N2"}


def cpu_model() -> str:
    """The host CPU's model name (x86: "model name"; Arm: implementer and part numbers)."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    for key in ("model name", "cpu model", "hardware"):
        if key in fields:
            return fields[key]
    if "cpu implementer" in fields and "cpu part" in fields:
        try:
            imp, part = int(fields["cpu implementer"], 16), int(fields["cpu part"], 16)
            name = _ARM_PARTS.get((imp, part), "Arm")
            return f"{name} (implementer 0x{imp:02x}, part 0x{part:03x})"
        except ValueError:
            pass
    return platform.processor() or platform.machine()


def prepare_unit(case, b: int, j: int):
    """Compact oracle call for query token (b, j) of `case` (a workloads.DecodeCase)."""
    import workloads
    L = int(case.seq_lens[b])
    idx = case.topk_indices[b, j].astype(np.int64)
    K = idx.size
    pages = -(-K // 64)
    ok = attention.valid_entries(idx, L, L - case.Q + j, case.page_table[b], case.num_pages)
    phys = np.where(ok, case.page_table[b][np.clip(idx // 64, 0, case.page_table.shape[1] - 1)].astype(np.int64) * 64
                    + idx % 64, -1)
    lat = np.zeros((pages * 64, 512), np.uint16)
    rope = np.zeros((pages * 64, 64), np.uint16)
    sel = np.nonzero(ok)[0]
    if sel.size:
        need = np.unique(phys[sel] // 64)
        plat, prope = workloads.host_rows(case, need)
        where = {int(p): i for i, p in enumerate(need)}
        src = np.array([where[int(p // 64)] * 64 + int(p % 64) for p in phys[sel]], np.int64)
        lat[sel] = plat[src]
        rope[sel] = prope[src]
    cache = pack.encode_rows(lat, rope).reshape(pages, 64, 352)
    # entry i of the list sits at compact position i; unusable entries stay unusable (-1)
    topk = np.where(ok, np.arange(K), -1).astype(np.int32).reshape(1, 1, K)
    return (case.q_bits[b:b + 1, j:j + 1].copy(), cache, np.arange(pages, dtype=np.int32)[None],
            topk, np.array([pages * 64], np.int32), case.softmax_scale)


def run_unit(u):
    q, cache, pt, tk, sl, scale = u
    return attention.sparse_decode(q, cache, pt, tk, sl, scale)


def _init(units):
    global _UNITS
    _UNITS = units


def _run_index(i):
    out, lse = run_unit(_UNITS[i])
    return float(np.nansum(lse))


def _time_indices(idx):
    t0 = time.perf_counter()
    for i in idx:
        run_unit(_UNITS[i])
    return time.perf_counter() - t0


def _prep_star(args):
    return prepare_unit(*args)


_ONE_THREAD = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _spawn_pool(workers, **kw):
    """A spawn-method pool whose workers run numpy's BLAS on one thread each (the limits must be in
    the environment when a worker starts, before numpy loads)."""
    saved = {k: os.environ.get(k) for k in _ONE_THREAD}
    os.environ.update({k: "1" for k in _ONE_THREAD})
    try:
        return mp.get_context("spawn").Pool(workers, **kw)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


class OraclePool:
    """A pool of `workers` spawned processes (one BLAS thread each) holding prepared units of one
    case, plus a one-process pool for the single-thread figure."""

    def __init__(self, case, units, workers: int):
        self.workers = max(1, int(workers))
        with _spawn_pool(self.workers) as p:
            prepared = p.map(_prep_star, [(case, b, j) for b, j in units])
        self.n = len(prepared)
        self.pool = _spawn_pool(self.workers, initializer=_init, initargs=(prepared,))
        self.single = _spawn_pool(1, initializer=_init, initargs=(prepared,))

    def step(self) -> float:
        """One pass over every prepared unit, spread over the workers; returns seconds."""
        t0 = time.perf_counter()
        self.pool.map(_run_index, range(self.n), chunksize=max(1, self.n // (4 * self.workers)))
        return time.perf_counter() - t0

    def step_single_thread(self, count: int) -> float:
        """The first `count` units one after another in one worker (one thread); returns seconds."""
        self.single.apply(_run_index, (0,))          # warm-up
        return self.single.apply(_time_indices, (list(range(min(count, self.n))),))

    def close(self):
        for p in (self.pool, self.single):
            p.close()
            p.join()
