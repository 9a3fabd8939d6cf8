#!/usr/bin/env python
"""Benchmark: one sparse MLA decode step over a paged NVFP4 cache on GB300.

Workload (the headline case): mixed agent batch, B=64 requests, Q=1 query token,
H=32 heads, context lengths uniform in [70K, 160K] tokens in 64-token pages from
one shared permuted pool, top-k = 2,048 positions per query. Synthetic seeded
data (workloads.make_case(2)); the cache (~2.6 GB) is packed on the device by
mla_kv_pack from device-drawn bf16 rows before timing.

A step is one sparse_mla_decode call (decode kernel + merge kernel). L2 is
flushed (256 MiB write) before every timed step; each step is timed with CUDA
events on the launching stream. The JSON line also carries:
  roofline     decode bytes at measured HBM bandwidth (the path is HBM-bound)
  e2e          the same step through the public call with pinned host buffers:
               the kernels read q / index lists / page table / lengths from host
               memory and write out + LSE back over NVLink-C2C, inside the timed
               region (the KV cache stays resident in HBM, as in serving)
  cpu_baseline the fp64 CPU oracle on a bounded sample of the same workload
  pack         mla_kv_pack of one 1M-row chunk of the cache fill (mean of 10 calls,
               L2 flushed before each), for context
--impl reference times the CPU oracle as the reference arm.
Multi-GPU (torchrun): every rank runs an independent replica (the path shards
by request with no exchange); the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse MLA decode µs/step & achieved HBM GB/s (% roofline), B=64, top-k 2048"
WORKLOAD = "mixed agent batch: B=64, Q=1, H=32, contexts U[70K,160K], 64-token pages, top-k 2048"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


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


def cpu_baseline_sample(units: int, seed: int = 0) -> dict:
    """Time the fp64 oracle (single thread) on `units` query tokens shaped like the
    headline workload (2,048 selected rows each, H=32); scaled to us per 64-token step."""
    code = r"""
import os, sys, time, json
sys.path.insert(0, %r)
import numpy as np
import workloads
from oracle import attention, pack
rng = np.random.default_rng(%d)
K, H, U = 2048, 32, %d
lat = workloads.f32_to_bf16_bits(rng.standard_normal((K, 512), dtype=np.float32))
rope = workloads.f32_to_bf16_bits(rng.standard_normal((K, 64), dtype=np.float32))
cache = pack.encode_rows(lat, rope).reshape(K // 64, 64, 352)
q = workloads.f32_to_bf16_bits(rng.standard_normal((1, 1, H, 576), dtype=np.float32))
pt = np.arange(K // 64, dtype=np.int32)[None]
sl = np.array([K], np.int32)
tks = [rng.permutation(K).astype(np.int32)[None, None] for _ in range(4)]
t0 = time.perf_counter()
for u in range(U):
    attention.sparse_decode(q, cache, pt, tks[u %% 4], sl, workloads.SOFTMAX_SCALE)
dt = time.perf_counter() - t0
print(json.dumps({"seconds": dt, "units": U}))
""" % (ROOT, seed, units)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    per_unit = d["seconds"] / d["units"]
    return {"value": per_unit * 64 * 1e6, "unit": "us/step", "cores": 1, "kind": "oracle",
            "sample": f"{d['units']} query tokens of the headline shape (2048 rows, H=32) through the fp64 "
                      f"oracle, single thread, scaled to one 64-token step; {d['seconds']:.1f} s of CPU work"}


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
    if rank != 0:
        return None
    steps, warm = args.steps, args.warmup
    # bounded sample per step: one query token (2,048 rows), scaled to the 64-token step
    per_step_units = 1
    if warm > 0:
        cpu_baseline_sample(warm)   # warm-up (imports, caches)
    t = cpu_baseline_sample(steps * per_step_units)
    value = t["value"]
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "us/step", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": value / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "one query token per step"},
        "cpu_baseline": {"value": value, "unit": "us/step", "cores": 1, "kind": "oracle", "sample": t["sample"]},
        "e2e": {"value": value, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_gpu(args, world, rank, local):
    import numpy as np
    import torch

    import nvfp4_compressed_sparse_gb300 as m
    import workloads

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    m.load_library()
    case = workloads.make_case(2)
    rows_total = case.num_pages * 64
    cache = torch.empty((case.num_pages, 64, 352), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # ---- fill the cache through mla_kv_pack in 1M-row chunks (device memory stays ~3 GB);
    # the pack of one chunk is timed for context (not the headline)
    chunk = 1 << 20
    pack_ms, pack_rows = None, 0
    for ci, s0 in enumerate(range(0, rows_total, chunk)):
        n = min(chunk, rows_total - s0)
        lat, rope = workloads.device_rows(case, n, dev, seed_offset=ci)
        slots = torch.arange(s0, s0 + n, device=dev)
        m.mla_kv_pack(lat, rope, slots, cache)
        if ci == 0:
            # mean of 10 calls on this chunk, L2 flushed (256 MiB write) before each
            flush0 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
            torch.cuda.synchronize(dev)
            times = []
            for _ in range(10):
                flush0.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                m.mla_kv_pack(lat, rope, slots, cache)
                e1.record(stream)
                times.append((e0, e1))
            torch.cuda.synchronize(dev)
            pack_ms, pack_rows = statistics.fmean(a.elapsed_time(b) for a, b in times), n
            del flush0
        del lat, rope, slots
    torch.cuda.synchronize(dev)
    pack_bytes = pack_rows * (1024 + 128 + 352 + 8)
    torch.cuda.empty_cache()

    q = torch.from_numpy(case.q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    pt = torch.from_numpy(case.page_table).to(dev)
    tk = torch.from_numpy(case.topk_indices).to(dev)
    sl = torch.from_numpy(case.seq_lens).to(dev)
    out = torch.empty((case.B, case.Q, case.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.B, case.Q, case.H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, m.sparse_mla_decode_workspace_size(case.B, case.Q, case.H, case.topk)),
                     dtype=torch.uint8, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    plan_ctas, plan_cluster = m.sparse_mla_decode_plan(case.B, case.Q, case.H, case.topk)
    launches_per_step = 1 if plan_cluster > 0 else 3
    timed_unit = ("sparse_mla_decode call (one cluster-mode decode kernel)" if plan_cluster > 0 else
                  "sparse_mla_decode call (q prep + decode + merge kernels)")

    def step():
        m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, out=out, lse=lse, workspace=ws,
                            dev_status=status, stream=stream)

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
        "config": {"workload": WORKLOAD, "B": case.B, "Q": case.Q, "H": case.H, "topk": case.topk,
                   "cache_pages": case.num_pages, "l2": "flushed before every step (256 MiB write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "achieved_hbm_gbs": achieved,
        "throughput_query_tokens_per_s": world * case.B * case.Q / t_s,
        "median_us_per_step": statistics.median(times_ms) * 1000.0,
        "roofline": {"bound": "hbm" if roof_hbm_us >= roof_tc_us else "tensor", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic_from_profile(),
                     "peak_kind": peak_kind, "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                     "roofline_us": max(roof_hbm_us, roof_tc_us), "tensor_roofline_us": roof_tc_us,
                     "timed_unit": timed_unit, "decode_ctas": plan_ctas, "cluster": plan_cluster},
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
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_sample(args.cpu_units)
    return result


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-units", type=int, default=320)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
