#!/usr/bin/env python
"""Benchmark: one sparse MLA decode step over a paged NVFP4 cache on GB300.

Workload (the headline case): mixed agent batch, B=64 requests, Q=1 query token,
H=32 heads, context lengths uniform in [70K, 160K] tokens in 64-token pages from
one shared permuted pool, top-k = 2,048 positions per query. Synthetic seeded
data (workloads.make_case(2)); the cache (~2.6 GB) is packed on the device by
mla_kv_pack from device-drawn bf16 rows before timing.

A step is one sparse_mla_decode call (q-prep, decode and merge kernels). L2 is
flushed (256 MiB write) before every timed step; each step is timed with CUDA
events on the launching stream. The JSON line also carries:
  roofline     decode bytes at the measured HBM bandwidth (the path is HBM-bound),
               and the same against the nominal 8 TB/s
  e2e          the same step through the public call with pinned host buffers:
               the kernels read q / index lists / page table / lengths from host
               memory and write out + LSE back over NVLink-C2C, inside the timed
               region (the KV cache stays resident in HBM, as in serving)
  cpu_baseline the fp64 CPU oracle on query tokens of the same workload (its own
               rows and index lists): one thread, and one process per host core
  configs      the decode-shard (B=16), spec-verify (192K-row pack + Q=4 decode in
               one step) and capacity (1.63M-token pool) cases, device-timed
  schedules    split vs cluster vs pair schedule for B = 1, 4, 16, 64 (headline requests)
  pack         mla_kv_pack of one 1M-row chunk of the cache fill (mean of 10 calls,
               L2 flushed before each), for context
--impl reference times the CPU oracle as the reference arm: every step runs all 64
query tokens of the headline case through the oracle, one process per host core.
Multi-GPU (torchrun): every rank runs an independent replica (the path shards
by request with no exchange); the slowest rank's time is reported.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse MLA decode µs/step & achieved HBM GB/s (% roofline), B=64, top-k 2048"
WORKLOAD = "mixed agent batch: B=64, Q=1, H=32, contexts U[70K,160K], 64-token pages, top-k 2048"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
NOMINAL_HBM_GBS = 8000.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def algorithmic_cost(case):
    """Bytes and FLOPs one decode step must move / do (per the row format):
    per query token: K_valid*352 row bytes + K*4 index bytes + H*576*2 (q) +
    H*512*2 (out) + H*4 (LSE); FLOPs 2*H*K_valid*(576+512). K_valid counts the
    entries the kernel loads (in range, causal, on a valid page)."""
    import numpy as np
    nbytes = flops = 0
    for b in range(case.B):
        L = int(case.seq_lens[b])
        row = case.page_table[b].astype(np.int64)
        for j in range(case.Q):
            idx = case.topk_indices[b, j].astype(np.int64)
            ok = (idx >= 0) & (idx < L) & (idx <= L - case.Q + j)
            col = np.where(ok, idx // 64, 0)
            ok &= col < row.size
            pg = row[np.clip(col, 0, row.size - 1)]
            ok &= (pg >= 0) & (pg < case.num_pages)
            kv = int(ok.sum())
            nbytes += kv * 352 + case.topk * 4 + case.H * (576 * 2 + 512 * 2 + 4)
            flops += 2 * case.H * kv * (576 + 512)
    return nbytes, flops


def traffic_from_profile():
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    src = os.path.join(ROOT, "nvfp4_compressed_sparse_gb300", "csrc", "decode_kernel.cu")
    prof = os.path.join(ROOT, "profiles", "decode_kernel_mixed_agent_B64.md")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        vals = {}
        for line in open(prof):
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
        if vals.get("kernel_source_sha256_16") == sha:
            return int(vals["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_pool(case, units, workers):
    """Spawned oracle workers holding the prepared query tokens `units` of `case`."""
    from oracle import timing
    return timing.OraclePool(case, units, workers)


def cpu_baseline(case, sample_units: int = 16, single_units: int = 2) -> dict:
    """The fp64 oracle on `sample_units` query tokens of the case (its own rows and index lists):
    all of them over one process per host core, and `single_units` of them in one thread; both
    scaled to one step of the case (B*Q query tokens)."""
    from oracle import timing
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(7)
    units_all = [(b, j) for b in range(case.B) for j in range(case.Q)]
    pick = sorted(rng.choice(len(units_all), size=min(sample_units, len(units_all)), replace=False))
    pool = oracle_pool(case, [units_all[i] for i in pick], cores)
    try:
        pool.step()                                   # warm-up
        par = min(pool.step() for _ in range(2))
        one = pool.step_single_thread(single_units)
    finally:
        pool.close()
    n = len(pick)
    scale = len(units_all)
    return {"value": par / n * scale * 1e6, "unit": "us/step", "cores": cores, "kind": "oracle",
            "cpu_model": timing.cpu_model(), "os_cpu_count": cores,
            "single_thread_us_per_step": one / single_units * scale * 1e6,
            "sample": f"{n} of the {scale} query tokens of this workload (own rows and index lists) through the "
                      f"fp64 oracle, one process per core ({cores}), scaled to one {scale}-token step; the single-"
                      f"thread figure runs {single_units} of them in one process"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step runs all B*Q query tokens of the headline case
    (its own rows and index lists) through the fp64 oracle, one process per host core."""
    if rank != 0:
        return None
    import workloads
    from oracle import timing
    case = workloads.make_case(2)
    cores = os.cpu_count() or 1
    units = [(b, j) for b in range(case.B) for j in range(case.Q)]
    full = len(units)
    if 0 < args.ref_units < full:
        units = units[:args.ref_units]
    pool = oracle_pool(case, units, cores)
    try:
        for _ in range(args.warmup):
            pool.step()
        wall0 = time.perf_counter()
        times = [pool.step() for _ in range(args.steps)]
        wall = time.perf_counter() - wall0
    finally:
        pool.close()
    mean_s = statistics.fmean(times) * full / len(units)
    value = mean_s * 1e6
    if len(units) == full:
        sample = (f"all {full} query tokens of the headline case per step (own rows and index lists), "
                  f"fp64 oracle, one process per core ({cores})")
    else:
        sample = (f"{len(units)} of the {full} query tokens per step, scaled to the full step, fp64 oracle, "
                  f"one process per core ({cores})")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": case.B, "Q": case.Q, "H": case.H, "topk": case.topk},
        "cpu_baseline": {"value": value, "unit": "us/step", "cores": cores, "kind": "oracle",
                         "cpu_model": timing.cpu_model(), "os_cpu_count": cores, "sample": sample},
        "e2e": {"value": value, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s_timed_region": wall,
    }


def fill_cache(m, workloads, case, dev, timed_pack=None):
    """Pack the case's whole cache on the device (1M-row chunks of device-drawn bf16 rows). With
    timed_pack = (stream, flush), the pack of the first chunk is also timed (mean of 10 calls, L2
    flushed before each) and (ms, rows) is returned with the cache."""
    import torch
    rows_total = case.num_pages * 64
    cache = torch.empty((case.num_pages, 64, 352), dtype=torch.uint8, device=dev)
    chunk = 1 << 20
    pack_ms, pack_rows = None, 0
    for ci, s0 in enumerate(range(0, rows_total, chunk)):
        n = min(chunk, rows_total - s0)
        lat, rope = workloads.device_rows(case, n, dev, seed_offset=ci)
        slots = torch.arange(s0, s0 + n, device=dev)
        m.mla_kv_pack(lat, rope, slots, cache)
        if ci == 0 and timed_pack is not None:
            stream, flush = timed_pack
            torch.cuda.synchronize(dev)
            times = []
            for _ in range(10):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                m.mla_kv_pack(lat, rope, slots, cache)
                e1.record(stream)
                times.append((e0, e1))
            torch.cuda.synchronize(dev)
            pack_ms, pack_rows = statistics.fmean(a.elapsed_time(b) for a, b in times), n
        del lat, rope, slots
    torch.cuda.synchronize(dev)
    return cache, pack_ms, pack_rows


def device_inputs(case, dev):
    import torch
    q = torch.from_numpy(case.q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    return (q, torch.from_numpy(case.page_table).to(dev), torch.from_numpy(case.topk_indices).to(dev),
            torch.from_numpy(case.seq_lens).to(dev))


def time_decode(m, case, cache, inputs, stream, flush, steps, warmup, cluster=None, pre=None):
    """Mean device time (ms) of one decode call (plus `pre`, a callable enqueued before it, timed
    separately), L2 flushed before each step. Returns (decode ms, pre ms or None)."""
    import torch
    q, pt, tk, sl = inputs
    out = torch.empty((case.B, case.Q, case.H, 512), dtype=torch.bfloat16, device=cache.device)
    lse = torch.empty((case.B, case.Q, case.H), dtype=torch.float32, device=cache.device)
    ws = torch.empty(max(1, m.sparse_mla_decode_workspace_size(case.B, case.Q, case.H, case.topk)),
                     dtype=torch.uint8, device=cache.device)
    ev = []
    for i in range(warmup + steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        if pre is not None:
            pre()
        e[1].record(stream)
        m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, out=out, lse=lse, workspace=ws,
                            stream=stream, cluster=cluster)
        e[2].record(stream)
        if i >= warmup:
            ev.append(e)
    torch.cuda.synchronize(cache.device)
    dec = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev)
    pre_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) if pre is not None else None
    return dec, pre_ms


def roofline_entry(nbytes, flops, ms, hbm):
    t = ms * 1e-3
    return {"us": ms * 1e3, "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / t / 1e9,
            "frac_of_measured_hbm": nbytes / t / 1e9 / hbm, "frac_of_nominal_hbm": nbytes / t / 1e9 / NOMINAL_HBM_GBS,
            "algorithmic_flops": flops}


def extra_configs(m, workloads, dev, stream, flush, hbm, steps):
    """Device-timed µs and roofline fractions of the decode-shard, spec-verify and capacity cases."""
    import torch
    res = {}
    for cfg in (1, 3, "3s", 4):
        case = workloads.make_case(cfg)
        cache, _, _ = fill_cache(m, workloads, case, dev)
        inputs = device_inputs(case, dev)
        nbytes, flops = algorithmic_cost(case)
        entry = {"name": workloads.CONFIG_NAMES[cfg], "B": case.B, "Q": case.Q, "H": case.H, "topk": case.topk,
                 "cluster": m.sparse_mla_decode_plan(case.B, case.Q, case.H, case.topk)[1]}
        if cfg == 3:
            # the step also packs the 6,000 new rows of every request (192K rows) into fresh pages
            n_new = case.new_slots.size
            lat, rope = workloads.device_rows(case, n_new, dev, seed_offset=99)
            slots = torch.from_numpy(case.new_slots).to(dev)
            pre = lambda: m.mla_kv_pack(lat, rope, slots, cache, stream=stream)
            dec_ms, pack_ms = time_decode(m, case, cache, inputs, stream, flush, steps, 5, pre=pre)
            pack_bytes = n_new * (1024 + 128 + 352 + 8)
            entry["decode"] = roofline_entry(nbytes, flops, dec_ms, hbm)
            entry["pack"] = {"rows": n_new, "us": pack_ms * 1e3, "algorithmic_bytes": pack_bytes,
                             "achieved_gbs": pack_bytes / (pack_ms * 1e-3) / 1e9,
                             "frac_of_measured_hbm": pack_bytes / (pack_ms * 1e-3) / 1e9 / hbm}
            entry["step_us"] = (dec_ms + pack_ms) * 1e3
            del lat, rope, slots
        else:
            dec_ms, _ = time_decode(m, case, cache, inputs, stream, flush, steps, 5)
            entry["decode"] = roofline_entry(nbytes, flops, dec_ms, hbm)
        if cfg == 4:
            entry["aliased_page_fraction"] = case.notes.get("aliased_fraction")
        if cfg in (3, "3s"):
            # distinct rows a request's query tokens select, against the entries of their lists
            uniq = [np.unique(case.topk_indices[b].reshape(-1)).size for b in range(case.B)]
            entry["distinct_rows_per_request"] = float(np.mean(uniq))
            entry["list_entries_per_request"] = case.Q * case.topk
        res[str(cfg)] = entry
        del cache, inputs
        torch.cuda.empty_cache()
    return res


def fp8_table(m, workloads, case, cache, dev, stream, flush, hbm, steps, native_ms):
    """The pages' three decode paths on the headline case, same rows: native (352-byte NVFP4
    rows), FP8 cache (576-byte FP8 rows packed from the same bf16 rows) and staged (NVFP4 rows
    copied to a 576-byte FP8 buffer, then the FP8 decode over it). Device µs per step and the
    algorithmic bytes per selected row each path moves through HBM."""
    import torch
    rows_total = case.num_pages * 64
    cache8 = torch.empty((case.num_pages, 64, 576), dtype=torch.uint8, device=dev)
    chunk = 1 << 20
    for ci, s0 in enumerate(range(0, rows_total, chunk)):
        n = min(chunk, rows_total - s0)
        lat, rope = workloads.device_rows(case, n, dev, seed_offset=ci)
        m.fp8_kv_pack(lat, rope, torch.arange(s0, s0 + n, device=dev), cache8)
        del lat, rope
    q, pt, tk, sl = device_inputs(case, dev)
    out = torch.empty((case.B, case.Q, case.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.B, case.Q, case.H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, m.sparse_mla_decode_workspace_size(case.B, case.Q, case.H, case.topk)),
                     dtype=torch.uint8, device=dev)
    staging = m.nvfp4_stage_fp8(cache, pt, tk, sl, stream=stream)
    staged, sidx, spt, ssl = staging
    qs = q.reshape(case.B * case.Q, 1, case.H, 576)
    out_s, lse_s = out.view(case.B * case.Q, 1, case.H, 512), lse.view(case.B * case.Q, 1, case.H)

    def timed(fns):
        ev = []
        for i in range(5 + steps):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
            e[0].record(stream)
            for k, fn in enumerate(fns):
                fn()
                e[k + 1].record(stream)
            if i >= 5:
                ev.append(e)
        torch.cuda.synchronize(dev)
        return [statistics.fmean(e[k].elapsed_time(e[k + 1]) for e in ev) * 1e3 for k in range(len(fns))]

    fp8_us, = timed([lambda: m.sparse_mla_decode_fp8(q, cache8, pt, tk, sl, case.softmax_scale, out=out, lse=lse,
                                                     workspace=ws, stream=stream)])
    del cache8
    torch.cuda.empty_cache()
    cache_t = torch.empty((case.num_pages, 64, 672), dtype=torch.uint8, device=dev)
    for ci, s0 in enumerate(range(0, rows_total, chunk)):
        n = min(chunk, rows_total - s0)
        lat, rope = workloads.device_rows(case, n, dev, seed_offset=ci)
        m.fp8_token_kv_pack(lat, rope, torch.arange(s0, s0 + n, device=dev), cache_t)
        del lat, rope
    tok_us, = timed([lambda: m.sparse_mla_decode_fp8_token(q, cache_t, pt, tk, sl, case.softmax_scale, out=out,
                                                           lse=lse, workspace=ws, stream=stream)])
    del cache_t
    torch.cuda.empty_cache()
    stage_us, staged_dec_us = timed([
        lambda: m.nvfp4_stage_fp8(cache, pt, tk, sl, staging=staging, stream=stream),
        lambda: m.sparse_mla_decode_fp8(qs, staged, spt, sidx, ssl, case.softmax_scale, out=out_s, lse=lse_s,
                                        workspace=ws, stream=stream)])
    n_rows = int(sum(min(int(case.seq_lens[b]), case.topk) for b in range(case.B))) * case.Q
    del staging, staged
    torch.cuda.empty_cache()
    return {
        "rows_selected": n_rows,
        "native": {"us": native_ms * 1e3, "bytes_per_row": 352},
        "fp8_cache": {"us": fp8_us, "bytes_per_row": 576},
        "fp8_per_token_cache": {"us": tok_us, "bytes_per_row": 672,
                                "format": "E4M3 latent / scale, bf16 rope / scale, fp32 scale per token"},
        "staged": {"us": stage_us + staged_dec_us, "stage_us": stage_us, "fp8_decode_us": staged_dec_us,
                   "bytes_per_row": 352 + 576 + 576},
        "pages_reference_gb200_us": {"native": 12.0, "staged": 17.7, "fp8": 13.7,
                                     "note": "the pages' numbers: 15 query tokens per launch on GB200"},
    }


def fold_table(m, workloads, dev, stream, flush, steps):
    """Query tokens folded over a shared index list (sparse_mla_decode_shared) against one pass per
    query token (sparse_mla_decode) on the same inputs: the spec-verify requests (B=32, contexts
    100K-156K) with 16 heads and Q = 2 or 4 draft tokens, each keeping 90 % of a shared set of 2,048
    positions. Device µs per step, L2 flushed before each step."""
    import torch
    base = workloads.make_case(3)
    cache, _, _ = fill_cache(m, workloads, base, dev)
    pt, sl = torch.from_numpy(base.page_table).to(dev), torch.from_numpy(base.seq_lens).to(dev)
    res = []
    for Q in (2, 4):
        rng = np.random.default_rng(4040 + Q)
        H, K = 16, base.topk
        qb = np.ascontiguousarray(base.q_bits[:, :Q, :H])
        q = torch.from_numpy(qb.view(np.int16)).to(dev).view(torch.bfloat16)
        lists = np.stack([workloads.subset_lists(rng, int(base.seq_lens[b]), Q, K, 0.9) for b in range(base.B)])
        shared, member = workloads.fold_lists(lists)
        tk = torch.from_numpy(lists.astype(np.int32)).to(dev)
        sh, mem = torch.from_numpy(shared).to(dev), torch.from_numpy(member).to(dev)
        out = torch.empty((base.B, Q, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((base.B, Q, H), dtype=torch.float32, device=dev)
        ws = torch.empty(max(m.sparse_mla_decode_workspace_size(base.B, Q, H, K),
                             m.sparse_mla_decode_workspace_size(base.B, 1, Q * H, shared.shape[1])),
                         dtype=torch.uint8, device=dev)
        times = {}
        for name, fn in (("per_token_us", lambda: m.sparse_mla_decode(q, cache, pt, tk, sl, base.softmax_scale,
                                                                        out=out, lse=lse, workspace=ws, stream=stream)),
                         ("folded_us", lambda: m.sparse_mla_decode_shared(q, cache, pt, sh, mem, sl,
                                                                          base.softmax_scale, out=out, lse=lse,
                                                                          workspace=ws, stream=stream))):
            ev = []
            for i in range(5 + steps):
                flush.zero_()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                e[0].record(stream)
                fn()
                e[1].record(stream)
                if i >= 5:
                    ev.append(e)
            torch.cuda.synchronize(dev)
            times[name] = statistics.fmean(a.elapsed_time(b) for a, b in ev) * 1e3
        res.append({"B": base.B, "Q": Q, "H": H, "list_entries_per_token": int(round(0.9 * K)),
                    "shared_list_len": int(shared.shape[1]), "heads_per_pass": min(32, Q * H), **times,
                    "speedup": times["per_token_us"] / times["folded_us"]})
    del cache
    torch.cuda.empty_cache()
    return res


def topk_table(m, case, cache, dev, stream, flush, hbm, steps):
    """indexer_topk on the headline case's query tokens (seeded N(0,1) fp32 logits over each causal
    range), alone and followed by sparse_mla_decode on the same stream. Algorithmic bytes: every
    logit in range read once plus the index lists written."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    S = (int(case.seq_lens.max()) + 3) // 4 * 4
    logits = torch.randn((case.B, case.Q, S), generator=g, device=dev, dtype=torch.float32)
    q, pt, _, sl = device_inputs(case, dev)
    idx = torch.empty((case.B, case.Q, case.topk), dtype=torch.int32, device=dev)
    out = torch.empty((case.B, case.Q, case.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.B, case.Q, case.H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, m.sparse_mla_decode_workspace_size(case.B, case.Q, case.H, case.topk)),
                     dtype=torch.uint8, device=dev)
    res = {}
    for name, with_decode in (("topk", False), ("topk_then_decode", True)):
        ev = []
        for i in range(5 + steps):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record(stream)
            m.indexer_topk(logits, sl, case.topk, out=idx, stream=stream)
            if with_decode:
                m.sparse_mla_decode(q, cache, pt, idx, sl, case.softmax_scale, out=out, lse=lse, workspace=ws,
                                    stream=stream)
            e[1].record(stream)
            if i >= 5:
                ev.append(e)
        torch.cuda.synchronize(dev)
        res[name + "_us"] = statistics.fmean(a.elapsed_time(b) for a, b in ev) * 1e3
    in_range = sum(max(0, min(int(case.seq_lens[b]) - case.Q + j + 1, S)) for b in range(case.B)
                   for j in range(case.Q))
    nbytes = 4 * in_range + 4 * case.B * case.Q * case.topk
    t = res["topk_us"] * 1e-6
    res.update({"rows": case.B * case.Q, "topk": case.topk, "logits": "N(0,1) fp32, seeded",
                "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / t / 1e9,
                "frac_of_measured_hbm": nbytes / t / 1e9 / hbm,
                "launches": "one 2-CTA cluster per query row (128 of the SMs; min(8, SMs / rows) CTAs per row)"})
    return res


def schedule_table(m, workloads, case, cache, dev, stream, flush, steps):
    """Split vs cluster schedule (forced wherever one wave of clusters fits) vs pair schedule for the
    first B requests of the headline case; cluster_size 0 = no wave of clusters fits."""
    import copy
    res = []
    for B in (1, 4, 16, 64):
        c = copy.copy(case)
        c.B = B
        c.seq_lens, c.page_table, c.topk_indices, c.q_bits = (case.seq_lens[:B], case.page_table[:B],
                                                             case.topk_indices[:B], case.q_bits[:B])
        inputs = device_inputs(c, dev)
        split_ms, _ = time_decode(m, c, cache, inputs, stream, flush, steps, 5, cluster=False)
        ctas, g = m.sparse_mla_decode_plan(c.B, c.Q, c.H, c.topk, cluster="any")
        row = {"B": B, "split_us": split_ms * 1e3,
               "split_ctas": m.sparse_mla_decode_plan(c.B, c.Q, c.H, c.topk, cluster=False)[0], "cluster_size": g,
               "default_cluster_size": m.sparse_mla_decode_plan(c.B, c.Q, c.H, c.topk)[1]}
        if g > 0:
            cl_ms, _ = time_decode(m, c, cache, inputs, stream, flush, steps, 5, cluster="any")
            row["cluster_us"] = cl_ms * 1e3
            row["cluster_ctas"] = ctas
        pair_ctas, pair_g = m.sparse_mla_decode_plan(c.B, c.Q, c.H, c.topk, cluster="pair")
        if pair_g == -2:
            pair_ms, _ = time_decode(m, c, cache, inputs, stream, flush, steps, 5, cluster="pair")
            row["pair_us"] = pair_ms * 1e3
            row["pair_ctas"] = pair_ctas
        res.append(row)
    return res


def run_gpu(args, world, rank, local):
    import torch

    import nvfp4_compressed_sparse_gb300 as m
    import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    m.load_library()
    case_id = int(args.case) if args.case.isdigit() else args.case
    case = workloads.make_case(case_id)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cache, pack_ms, pack_rows = fill_cache(m, workloads, case, dev, timed_pack=(stream, flush))
    pack_bytes = pack_rows * (1024 + 128 + 352 + 8)
    torch.cuda.empty_cache()

    q, pt, tk, sl = device_inputs(case, dev)
    out = torch.empty((case.B, case.Q, case.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.B, case.Q, case.H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, m.sparse_mla_decode_workspace_size(case.B, case.Q, case.H, case.topk)),
                     dtype=torch.uint8, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)

    schedule = {"default": None, "split": False, "pair": "pair"}[args.schedule]
    plan_ctas, plan_cluster = m.sparse_mla_decode_plan(case.B, case.Q, case.H, case.topk, cluster=schedule)
    launches_per_step = 1 if plan_cluster > 0 else 3
    timed_unit = ("sparse_mla_decode call (one cluster-mode decode kernel)" if plan_cluster > 0 else
                  "sparse_mla_decode call (q prep + pair decode + merge kernels)" if plan_cluster == -2 else
                  "sparse_mla_decode call (q prep + decode + merge kernels)")

    def step():
        m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, out=out, lse=lse, workspace=ws,
                            dev_status=status, stream=stream, cluster=schedule)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_ms = statistics.fmean(times_ms)
    mean_ms = max_over_ranks(mean_ms, world)
    st = status.cpu().tolist()

    # ---- end to end through the public call with host buffers: q, page table, index lists and
    # lengths in pinned host memory, out and LSE written to pinned host memory. The kernels move
    # those bytes over the host link themselves, inside each timed step.
    hq = torch.empty_like(q, device="cpu").pin_memory()
    hq.copy_(q)
    hpt, htk, hsl = pt.cpu().pin_memory(), tk.cpu().pin_memory(), sl.cpu().pin_memory()
    hout = torch.empty_like(out, device="cpu").pin_memory()
    hlse = torch.empty_like(lse, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hpt, htk, hsl))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()

    def host_step():
        m.sparse_mla_decode(hq, cache, hpt, htk, hsl, case.softmax_scale, out=hout, lse=hlse, workspace=ws,
                            dev_status=status, stream=stream)

    Ke = max(1, min(K, 500))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    for i in range(Ke + 3):
        flush.zero_()
        if i >= 3:
            es[i - 3].record(stream)
        host_step()
        if i >= 3:
            ee[i - 3].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = statistics.fmean(s.elapsed_time(e) for s, e in zip(es, ee))
    e2e_ms = max_over_ranks(e2e_ms, world)
    step()
    torch.cuda.synchronize(dev)
    e2e_same = bool(torch.equal(out.cpu(), hout) and torch.equal(lse.cpu(), hlse))

    nbytes, flops = algorithmic_cost(case)
    hbm, tflops, peak_kind = peaks()
    t_s = mean_ms * 1e-3
    achieved = nbytes / t_s / 1e9
    roof_hbm_us = nbytes / (hbm * 1e9) * 1e6
    roof_tc_us = flops / (tflops * 1e12) * 1e6
    result = {
        "metric": METRIC, "value": mean_ms * 1000.0, "unit": "us/step", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD if case_id == 2 else workloads.CONFIG_NAMES[case_id], "B": case.B,
                   "Q": case.Q, "H": case.H, "topk": case.topk,
                   "cache_pages": case.num_pages, "l2": "flushed before every step (256 MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "achieved_hbm_gbs": achieved,
        "throughput_query_tokens_per_s": world * case.B * case.Q / t_s,
        "median_us_per_step": statistics.median(times_ms) * 1000.0,
        "roofline": {"bound": "hbm" if roof_hbm_us >= roof_tc_us else "tensor", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic_from_profile() if plan_cluster != -2 else None,
                     "peak_kind": peak_kind, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                     "roofline_us": max(roof_hbm_us, roof_tc_us), "tensor_roofline_us": roof_tc_us,
                     "timed_unit": timed_unit, "decode_ctas": plan_ctas, "cluster": plan_cluster,
                     "schedule": args.schedule},
        "e2e": {"value": e2e_ms * 1000.0, "unit": "us/step", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "transfer": "kernels read q / page table / index lists / lengths from pinned host memory and write "
                            "out + LSE to pinned host memory (NVLink-C2C), inside each timed step",
                "bitwise_equal_to_device_buffers": e2e_same},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "pack": {"rows": pack_rows, "us": pack_ms * 1000.0, "gbs": pack_bytes / (pack_ms * 1e-3) / 1e9,
                 "frac_of_hbm": pack_bytes / (pack_ms * 1e-3) / 1e9 / hbm},
        "dev_status": st,
        "wall_s_timed_region": wall,
    }
    if not args.no_extra and world == 1 and case_id == 2:
        result["schedules"] = schedule_table(m, workloads, case, cache, dev, stream, flush, min(K, 200))
        result["indexer_topk"] = topk_table(m, case, cache, dev, stream, flush, hbm, min(K, 200))
        result["fp8_paths"] = fp8_table(m, workloads, case, cache, dev, stream, flush, hbm, min(K, 200), mean_ms)
        del cache, hq, hpt, htk, hsl, hout, hlse, ws
        torch.cuda.empty_cache()
        result["configs"] = extra_configs(m, workloads, dev, stream, flush, hbm, min(K, 200))
        result["fold"] = fold_table(m, workloads, dev, stream, flush, min(K, 200))
    if rank == 0 and world == 1 and not args.no_cpu_baseline and case_id == 2:
        result["cpu_baseline"] = cpu_baseline(case)
    return result


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the extra cases and the schedule table")
    ap.add_argument("--schedule", default="default", choices=["default", "split", "pair"],
                    help="decode schedule of the timed step (default: the library's; pair: NVFP4MLA_FLAG_PAIR). "
                         "The end-to-end leg, with results in host memory, always runs the split schedule.")
    ap.add_argument("--case", default="2", choices=["0", "1", "2", "3", "3s", "4"],
                    help="workload of the timed line (default 2, the headline; the others for profiling, "
                         "without the extra tables)")
    ap.add_argument("--ref-units", type=int, default=0,
                    help="reference arm: query tokens per step (0 = all of the headline case)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_gpu(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
