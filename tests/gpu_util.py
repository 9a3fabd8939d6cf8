"""Helpers shared by the GPU parity tests (device transfer of seeded inputs,
oracle evaluation of sampled units)."""
import numpy as np
import torch

import workloads
from oracle import attention, codec, pack

OUT_ATOL, OUT_RTOL, LSE_ATOL = 2e-3, 1e-2, 1e-3


def bf16_dev(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def decode_inputs(case, dev="cuda"):
    return (bf16_dev(case.q_bits, dev), i32(case.page_table, dev), i32(case.topk_indices, dev),
            i32(case.seq_lens, dev))


def assert_close(out, lse, ref_out, ref_lse, what=""):
    o = out.float().cpu().numpy() if isinstance(out, torch.Tensor) else out
    l = lse.cpu().numpy() if isinstance(lse, torch.Tensor) else lse
    err = np.abs(o - ref_out) - (OUT_ATOL + OUT_RTOL * np.abs(ref_out))
    assert np.all(err <= 0), f"{what}: out outside tolerance, worst excess {err.max():.3e}"
    both_inf = np.isneginf(l) & np.isneginf(ref_lse)
    d = np.where(both_inf, 0.0, np.abs(l - ref_lse))
    assert np.all(d <= LSE_ATOL), f"{what}: lse outside tolerance, worst {np.nanmax(d):.3e}"


def oracle_units_from_device_rows(case, units, lat_dev, rope_dev, fmt="nvfp4"):
    """Oracle outputs for (b, j) units, encoding the selected rows from their bf16
    inputs (gathered from the device input tensors by physical slot) in the cache format
    fmt ("nvfp4", "fp8", "staged" or "token"). The CPU work runs in a pool of spawned worker
    processes."""
    from tests import oracle_pool
    keys, jobs = [], []
    for b, j in units:
        L = int(case.seq_lens[b])
        idx = case.topk_indices[b, j].astype(np.int64)
        ok = attention.valid_entries(idx, L, L - case.Q + j, case.page_table[b], case.num_pages)
        sel = idx[ok]
        slots = case.page_table[b][sel // 64].astype(np.int64) * 64 + sel % 64
        st = torch.from_numpy(slots).to(lat_dev.device)
        jobs.append((case.q_bits[b, j], bits_of(lat_dev[st]), bits_of(rope_dev[st]), case.softmax_scale, fmt))
        keys.append((b, j))
    return dict(zip(keys, oracle_pool.attend_units(jobs)))
