"""sparse_mla_decode_noalloc: the decode step for callers that cannot allocate
device memory (an operator inside an engine that owns all device memory, a
plugin without a workspace argument). It must give the same results as
sparse_mla_decode, on consecutive calls that share its built-in scratch.

This file is collected last on purpose: if it fails, a run stopped at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import pack
from tests.gpu_util import OUT_ATOL, OUT_RTOL, LSE_ATOL, bf16_dev, decode_inputs

pytestmark = pytest.mark.gpu

V = ctypes.c_void_p


def _noalloc_fn():
    lib = m.load_library()
    fn = lib.sparse_mla_decode_noalloc
    fn.argtypes = [V, V, ctypes.c_int64, V, ctypes.c_int64, V, V, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_float, V, V, V, ctypes.c_uint32, V]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, q, cache, pt, tk, sl, case, out, lse, flags=0):
    return fn(V(q.data_ptr()), V(cache.data_ptr()), cache.shape[0], V(pt.data_ptr()), pt.shape[1],
              V(tk.data_ptr()), V(sl.data_ptr()), case.B, case.Q, case.H, case.topk,
              ctypes.c_float(case.softmax_scale), V(out.data_ptr()), V(lse.data_ptr()), None, flags,
              V(torch.cuda.current_stream().cuda_stream))


def _case_on_device(spec, seed):
    case = workloads.small_case(seed=seed, **spec)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(case.num_pages * 64, device="cuda"), cache)
    return case, cache


def _assert_close(out, lse, ref_out, ref_lse):
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    ro, rl = ref_out.float().cpu().numpy(), ref_lse.cpu().numpy()
    assert np.all(np.abs(o - ro) <= OUT_ATOL + OUT_RTOL * np.abs(ro))
    same_inf = np.isneginf(l) & np.isneginf(rl)
    assert np.all(np.where(same_inf, 0.0, np.abs(l - rl)) <= LSE_ATOL)


@pytest.mark.parametrize("spec", [dict(B=3, Q=2, H=32, topk=700, L=(3000, 2600, 900), invalid_frac=0.1),
                                  dict(B=2, Q=1, H=64, topk=300, L=(1200, 800))])
def test_noalloc_matches_regular_entry_point_twice(spec):
    fn = _noalloc_fn()
    case = workloads.small_case(seed=31, **spec)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(case.num_pages * 64, device="cuda"), cache)
    q, pt, tk, sl = decode_inputs(case)
    ref_out, ref_lse = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale)
    torch.cuda.synchronize()
    ro, rl = ref_out.float().cpu().numpy(), ref_lse.cpu().numpy()
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _call(fn, q, cache, pt, tk, sl, case, out, lse) == 0
        torch.cuda.synchronize()
        o, l = out.float().cpu().numpy(), lse.cpu().numpy()
        assert np.all(np.abs(o - ro) <= OUT_ATOL + OUT_RTOL * np.abs(ro))
        same_inf = np.isneginf(l) & np.isneginf(rl)
        assert np.all(np.where(same_inf, 0.0, np.abs(l - rl)) <= LSE_ATOL)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _noalloc_fn()
    need = m.sparse_mla_decode_workspace_size(4096, 16, 128, 8192)
    assert need > (32 << 20)
    big = workloads.small_case(B=1, Q=1, H=32, topk=10, L=(64,), seed=2)
    big.B, big.Q, big.H, big.topk = 4096, 16, 128, 8192
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    d = dummy.data_ptr()
    rc = fn(V(d), V(d), 1, V(d), 1, V(d), V(d), big.B, big.Q, big.H, big.topk, ctypes.c_float(0.07), V(d), V(d),
            None, 0, None)
    assert rc == 4      # NVFP4MLA_ERR_WORKSPACE, returned before anything is enqueued


def test_noalloc_later_calls_take_no_device_memory():
    """After the first call on the device, calls of other shapes, flags and buffer kinds leave
    the device's free memory unchanged: the scratch is the library's static region, and the
    call allocates nothing (every input and output below is allocated before the first call)."""
    fn = _noalloc_fn()
    specs = [dict(B=2, Q=1, H=32, topk=500, L=(3000, 2500)), dict(B=1, Q=2, H=16, topk=200, L=(900,)),
             dict(B=3, Q=1, H=64, topk=129, L=(700, 800, 900))]
    prepared = []
    for i, spec in enumerate(specs):
        case, cache = _case_on_device(spec, seed=40 + i)
        q, pt, tk, sl = decode_inputs(case)
        out = torch.empty((case.B, case.Q, case.H, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((case.B, case.Q, case.H), dtype=torch.float32, device="cuda")
        prepared.append((case, cache, q, pt, tk, sl, out, lse))
    # one pass over every shape and flag first: the first call looks up the scratch address, and
    # CUDA loads each kernel on its first launch (module loading, not this entry point)
    for rnd in range(2):
        if rnd == 1:
            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
        for flags in (0, m.FLAG_CLUSTER, 3):
            for case, cache, q, pt, tk, sl, out, lse in prepared:
                assert _call(fn, q, cache, pt, tk, sl, case, out, lse, flags) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


@pytest.mark.parametrize("mode", ["cluster", "host-results"])
def test_noalloc_cluster_schedule_and_host_results(mode):
    """The cluster schedule on the shared scratch, and results written to page-locked host
    memory (the polling merge, whose tags live in the scratch), against the regular entry
    point, on two calls in a row."""
    fn = _noalloc_fn()
    spec = dict(B=2, Q=1, H=32, topk=1024, L=(3000, 2600)) if mode == "cluster" else \
        dict(B=3, Q=2, H=32, topk=300, L=(1500, 2000, 900))
    case, cache = _case_on_device(spec, seed=51)
    q, pt, tk, sl = decode_inputs(case)
    cluster = mode == "cluster"
    if cluster:
        assert m.sparse_mla_decode_plan(case.B, case.Q, case.H, case.topk, cluster=True)[1] >= 1
    ref_out, ref_lse = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, cluster=cluster)
    torch.cuda.synchronize()
    for _ in range(2):
        if mode == "host-results":
            out = torch.full(tuple(ref_out.shape), float("nan"), dtype=torch.bfloat16).pin_memory()
            lse = torch.full(tuple(ref_lse.shape), float("nan"), dtype=torch.float32).pin_memory()
        else:
            out = torch.full_like(ref_out, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
        assert _call(fn, q, cache, pt, tk, sl, case, out, lse, m.FLAG_CLUSTER if cluster else 0) == 0
        torch.cuda.synchronize()
        _assert_close(out, lse, ref_out, ref_lse)
