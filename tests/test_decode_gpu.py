"""sparse_mla_decode on the GPU vs the CPU oracle.

Outputs within |out - ref| <= 2e-3 + 1e-2 |ref| and |lse - ref| <= 1e-3, where
the reference is fp64 attention over the same dequantised cache; index and page
handling bit-exact (bitwise invariance under page permutation, exact
single-token output, exact status counts)."""
import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import attention, pack
from tests.gpu_util import (assert_close, bf16_dev, bits_of, decode_inputs, i32,
                            oracle_units_from_device_rows)

pytestmark = pytest.mark.gpu


def _host_cache(case):
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    return lat, rope, rows


def _gpu_cache(lat, rope, num_pages):
    cache = torch.zeros((num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(num_pages * 64, device="cuda"), cache)
    return cache


def _decode(case, cache, **kw):
    q, pt, tk, sl = decode_inputs(case)
    out, lse = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, **kw)
    torch.cuda.synchronize()
    return out, lse


SMALL = [
    dict(B=2, Q=1, H=16, topk=200, L=(700, 1000)),                       # ragged tail: 128 + 72
    dict(B=2, Q=1, H=32, topk=300, L=(2000, 900)),
    dict(B=1, Q=4, H=32, topk=256, L=(3000,)),                            # causal across 4 query tokens
    dict(B=3, Q=2, H=64, topk=130, L=(500, 600, 700)),                    # two head groups
    dict(B=1, Q=1, H=128, topk=129, L=(400,)),                            # four head groups
    dict(B=2, Q=2, H=32, topk=384, L=(1500, 1400), invalid_frac=0.25, dup=True, causal_tail=True),
    dict(B=4, Q=1, H=16, topk=50, L=(40, 60, 2000, 64)),                  # short contexts leave -1 entries
    dict(B=2, Q=2, H=32, topk=256, L=(3000, 2600), shared=0.9),           # draft tokens sharing 90 % of rows
    dict(B=1, Q=4, H=16, topk=512, L=(5000,), shared=0.9),
    dict(B=2, Q=4, H=32, topk=300, L=(4000, 1900), shared=0.5),
]


def _spec_id(s):
    return "B{B}Q{Q}H{H}K{topk}".format(**s) + (f"S{s['shared']}" if "shared" in s else "")


@pytest.mark.parametrize("spec", SMALL, ids=_spec_id)
@pytest.mark.parametrize("max_ctas", [0, "split", 1, 3])
def test_small_cases_match_oracle(spec, max_ctas):
    case = workloads.small_case(seed=100 + len(str(spec)), **spec)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    np.testing.assert_array_equal(cache.cpu().numpy(), rows)
    kw = dict(cluster=False) if max_ctas == "split" else dict(max_ctas=max_ctas)   # 0: the default schedule
    out, lse = _decode(case, cache, **kw)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, f"{spec} max_ctas={max_ctas}")


# Cases the cluster schedule (NVFP4MLA_FLAG_CLUSTER) takes on a 152-SM GB300 (expected G in the id): one CTA per
# tile, several tiles per CTA, ragged tails, H=16 and several head groups, ranks whose tiles
# hold only unused (-1) entries, invalid and duplicate entries.
CLUSTER = [
    (1, dict(B=1, Q=1, H=32, topk=100, L=(900,))),
    (2, dict(B=1, Q=1, H=16, topk=256, L=(4096,))),
    (3, dict(B=2, Q=2, H=64, topk=384, L=(1500, 1400))),
    (3, dict(B=1, Q=1, H=16, topk=300, L=(100,))),                    # ranks 1, 2: only -1 entries
    (4, dict(B=2, Q=1, H=32, topk=500, L=(3000, 2500), invalid_frac=0.25, dup=True)),
    (5, dict(B=1, Q=1, H=32, topk=600, L=(5000,))),
    (6, dict(B=3, Q=1, H=16, topk=700, L=(900, 1200, 800))),
    (7, dict(B=1, Q=1, H=32, topk=833, L=(2000,))),
    (8, dict(B=1, Q=1, H=32, topk=1024, L=(1500,))),
    (8, dict(B=10, Q=1, H=32, topk=2048, L=(3000,) * 10)),          # two tiles per CTA
]


@pytest.mark.parametrize("G,spec", CLUSTER, ids=lambda x: x if isinstance(x, int) else
                         "B{B}Q{Q}H{H}K{topk}".format(**x))
def test_cluster_schedule_matches_oracle(G, spec):
    ctas, cluster = m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"], cluster=True)
    # default: the cluster schedule only for clusters of <= 2 CTAs that are at most two tiles per CTA
    # less balanced than the split; NVFP4MLA_FLAG_SPLIT: never
    default_g = m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"])[1]
    assert default_g in (0, cluster) and (default_g == 0 or default_g <= 2)
    assert m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"], cluster=False)[1] == 0
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert cluster == G, (ctas, cluster)
    else:
        assert cluster >= 1, (ctas, cluster)
    assert ctas == cluster * spec["B"] * spec["Q"] * max(1, spec["H"] // 32)
    assert m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"], max_ctas=152, cluster=True)[1] == 0
    case = workloads.small_case(seed=300 + G + spec["topk"], **spec)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    out, lse = _decode(case, cache, cluster=True)
    assert_close(out, lse, ref_out, ref_lse, f"cluster G={cluster} {spec}")
    out2, lse2 = _decode(case, cache, cluster=True)        # deterministic across calls
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_all_entries_unused_gives_zero_and_neg_inf():
    case = workloads.small_case(B=2, Q=1, H=32, topk=300, L=(500, 600), seed=3)
    case.topk_indices[:] = -1
    case.topk_indices[1, 0, 5] = 10**6          # past seq_len: also unused
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = _decode(case, cache, dev_status=status)
    assert bool((out == 0).all())
    assert bool(torch.isneginf(lse).all())
    assert status.cpu().tolist() == [1, 0, 0, 0]


def test_single_valid_entry_is_exact():
    case = workloads.small_case(B=1, Q=1, H=16, topk=128, L=(300,), seed=4)
    case.topk_indices[:] = -1
    case.topk_indices[0, 0, 77] = 201
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    out, lse = _decode(case, cache)
    c = attention.dequant_rows(rows[case.page_table[0][201 // 64], 201 % 64][None])[0]
    # the dequantised row is exact in bf16, so the output equals it exactly (as values: the sign of
    # a zero is not kept through fp32 accumulation)
    np.testing.assert_array_equal(out.float().cpu().numpy()[0, 0], np.broadcast_to(c[:512], (16, 512)))
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3


def test_deterministic_and_page_permutation_bitwise():
    case = workloads.small_case(B=2, Q=1, H=32, topk=500, L=(3000, 2500), seed=8)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    out1, lse1 = _decode(case, cache)
    out2, lse2 = _decode(case, cache)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    perm = np.random.default_rng(1).permutation(case.num_pages)
    cache_p = torch.empty_like(cache)
    cache_p[torch.from_numpy(perm).cuda()] = cache
    case_p = workloads.small_case(B=2, Q=1, H=32, topk=500, L=(3000, 2500), seed=8)
    case_p.page_table = np.where(case.page_table >= 0, perm[np.clip(case.page_table, 0, None)], -1).astype(np.int32)
    out3, lse3 = _decode(case_p, cache_p)
    assert torch.equal(out1, out3) and torch.equal(lse1, lse3)


def test_status_counts_bad_indices_and_pages():
    case = workloads.small_case(B=2, Q=2, H=64, topk=200, L=(900, 700), seed=12)
    tk = case.topk_indices
    tk[0, 0, :10] = 5000            # past seq_len            -> bad index
    tk[0, 1, 10:13] = -3            # negative, not -1        -> bad index
    tk[1, 0, 0:4] = 699             # past causal for j = 0   -> bad index
    tk[1, 1, 50:60] = -1            # unused                  -> not counted
    case.page_table[1, 2] = -1      # positions 128..191 of request 1 -> bad page
    case.page_table[0, 3] = 10**6   # positions 192..255 of request 0 -> bad page
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = _decode(case, cache, dev_status=status)
    bad_idx = bad_page = 0
    for b in range(2):
        L = int(case.seq_lens[b])
        for j in range(2):
            for idx in tk[b, j]:
                if idx == -1:
                    continue
                if idx < 0 or idx >= L or idx > L - 2 + j:
                    bad_idx += 1
                    continue
                pg = case.page_table[b][idx // 64]
                if pg < 0 or pg >= case.num_pages:
                    bad_page += 1
    assert status.cpu().tolist() == [bad_idx, bad_page, 0, 0]
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, tk, case.seq_lens,
                                               case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, "status case")


def test_two_streams_with_event_order():
    case = workloads.small_case(B=2, Q=1, H=32, topk=256, L=(1200, 1300), seed=21)
    lat, rope, rows = _host_cache(case)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    latd, roped = bf16_dev(lat), bf16_dev(rope)
    slots = torch.arange(case.num_pages * 64, device="cuda")
    q, pt, tk, sl = decode_inputs(case)
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        m.mla_kv_pack(latd, roped, slots, cache, stream=s1)
        ev = torch.cuda.Event()
        ev.record(s1)
    s2.wait_event(ev)
    with torch.cuda.stream(s2):
        out, lse = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, stream=s2)
    torch.cuda.synchronize()
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, "two streams")


def test_dense_control_equals_dense_oracle():
    case = workloads.make_case("4d")
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    out, lse = _decode(case, cache)
    ref_out, ref_lse = attention.dense_decode(case.q_bits, rows, case.page_table, case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, "dense control")


@pytest.mark.parametrize("schedule", ["default", "split"])
@pytest.mark.parametrize("cfg", [0, 1, 2, 3, "3s", 4])
def test_full_size_case_every_unit(cfg, schedule):
    """The five cases at full size, in the launch configuration the bench uses; the cache is
    packed on the device from device-drawn bf16 rows, and every query token is checked against
    the oracle (which re-encodes the selected rows from the same bf16 inputs), so every
    stream-K segment boundary and merge layout of the real schedule is covered."""
    case = workloads.make_case(cfg)
    rows_total = case.num_pages * 64
    lat, rope = workloads.device_rows(case, rows_total, "cuda")
    cache = torch.empty((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(lat, rope, torch.arange(rows_total, device="cuda"), cache)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = _decode(case, cache, dev_status=status, cluster=None if schedule == "default" else False)
    assert status.cpu().tolist() == [0, 0, 0, 0]
    units = [(b, j) for b in range(case.B) for j in range(case.Q)]
    ref = oracle_units_from_device_rows(case, units, lat, rope)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for (b, j), (ro, rl) in ref.items():
        assert_close(o[b, j], l[b, j], ro, rl, f"cfg {cfg} unit {(b, j)}")
    assert np.isfinite(o).all()


@pytest.mark.parametrize("kw", [dict(cluster=False), dict(max_ctas=1), dict(cluster=True)], ids=["split", "split-prep", "cluster"])
def test_pinned_host_buffers_match_device_buffers(kw):
    """q, page table, index lists, lengths, out and LSE in page-locked host memory (read and
    written by the kernels over the host link) give bitwise the device-buffer results."""
    case = workloads.small_case(B=3, Q=2, H=32, topk=300, L=(1500, 2000, 900), seed=21)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    q, pt, tk, sl = decode_inputs(case)
    out_d, lse_d = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, **kw)
    hq, hpt, htk, hsl = (t.cpu().pin_memory() for t in (q, pt, tk, sl))
    hout = torch.empty(tuple(out_d.shape), dtype=out_d.dtype).pin_memory()
    hlse = torch.empty(tuple(lse_d.shape), dtype=lse_d.dtype).pin_memory()
    m.sparse_mla_decode(hq, cache, hpt, htk, hsl, case.softmax_scale, out=hout, lse=hlse, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out_d.cpu(), hout) and torch.equal(lse_d.cpu(), hlse)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(hout, hlse, ref_out, ref_lse, f"host buffers {kw}")


@pytest.mark.parametrize("H", [16, 128])
def test_host_q_alone_matches_device_q(H):
    """q in page-locked host memory alone (its prep grid then splits every unit over a cluster of
    CTAs that share the unit's maximum): bitwise the device-q result, for one and several head
    groups."""
    case = workloads.small_case(B=2, Q=3, H=H, topk=260, L=(1300, 2100), seed=40 + H)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    q, pt, tk, sl = decode_inputs(case)
    out_d, lse_d = m.sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale)
    out_h, lse_h = m.sparse_mla_decode(q.cpu().pin_memory(), cache, pt, tk, sl, case.softmax_scale)
    torch.cuda.synchronize()
    assert torch.equal(out_d, out_h) and torch.equal(lse_d, lse_h)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(out_h, lse_h, ref_out, ref_lse, f"host q H={H}")


def test_pageable_host_memory_is_rejected_before_launch():
    import ctypes
    case = workloads.small_case(B=1, Q=1, H=32, topk=128, L=(900,), seed=5)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    q, pt, tk, sl = decode_inputs(case)
    pageable_q = q.cpu()
    with pytest.raises(ValueError):
        m.sparse_mla_decode(pageable_q, cache, pt, tk, sl, case.softmax_scale)
    lib = m.load_library()
    out = torch.full((1, 1, 32, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 1, 32), 7.0, dtype=torch.float32, device="cuda")
    wsb = m.sparse_mla_decode_workspace_size(1, 1, 32, 128)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    for name in ("q", "out", "cache"):
        args = dict(q=q, out=out, cache=cache)
        args[name] = args[name].cpu()               # pageable copy
        rc = lib.sparse_mla_decode(P(args["q"]), P(args["cache"]), case.num_pages, P(pt), pt.shape[1], P(tk), P(sl),
                                   1, 1, 32, 128, ctypes.c_float(case.softmax_scale), P(args["out"]), P(lse), P(ws),
                                   wsb, None, 0, None)
        assert rc == 1, (name, rc)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())   # nothing was launched


@pytest.mark.parametrize("spec", [dict(B=1, Q=1, H=32, topk=2048, L=(5000,)), dict(B=4, Q=1, H=32, topk=2048, L=(4000,) * 4),
                                  dict(B=3, Q=1, H=16, topk=1000, L=(3000, 1200, 2500))],
                         ids=lambda s: "B{B}H{H}K{topk}".format(**s))
def test_cluster_any_schedule_matches_oracle(spec):
    """NVFP4MLA_FLAG_CLUSTER_ANY: the cluster schedule wherever one wave of clusters fits, including
    shapes where a CTA then runs more tiles than under the split schedule (the schedule table of the
    benchmark uses it)."""
    ctas, g = m.sparse_mla_decode_plan(spec["B"], spec["Q"], spec["H"], spec["topk"], cluster="any")
    assert g >= 1 and ctas == g * spec["B"] * spec["Q"] * max(1, spec["H"] // 32)
    case = workloads.small_case(seed=77 + spec["B"], **spec)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    out, lse = _decode(case, cache, cluster="any")
    assert_close(out, lse, ref_out, ref_lse, f"cluster any G={g} {spec}")


@pytest.mark.parametrize("spec,kw", [
    (dict(B=2, Q=1, H=32, topk=8192, L=(20000, 12000)), {}),                 # the largest index list: 64 tiles
    (dict(B=2, Q=1, H=32, topk=8192, L=(20000, 12000)), dict(cluster="pair")),
    (dict(B=1, Q=16, H=128, topk=300, L=(5000,)), {}),                       # the most query tokens, 4 head groups
    (dict(B=2, Q=16, H=32, topk=2048, L=(9000, 3000)), dict(max_ctas=5)),   # 16 causal ranges per request
], ids=["K8192", "K8192-pair", "Q16H128", "Q16-5ctas"])
def test_maximum_sizes_match_oracle(spec, kw):
    """The limits the C ABI accepts: top-k = NVFP4MLA_MAX_TOPK and Q = 16 query tokens per request."""
    case = workloads.small_case(seed=900 + spec["Q"] + spec["topk"], **spec)
    lat, rope, rows = _host_cache(case)
    cache = _gpu_cache(lat, rope, case.num_pages)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = _decode(case, cache, dev_status=status, **kw)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, case.topk_indices,
                                               case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, f"{spec} {kw}")
    bad = 0
    for b in range(case.B):
        L = int(case.seq_lens[b])
        for j in range(case.Q):
            tk = case.topk_indices[b, j]
            bad += int(np.sum((tk != -1) & ((tk < 0) | (tk >= L) | (tk > L - case.Q + j))))
    assert status.cpu().tolist()[0] == bad and status.cpu().tolist()[1:] == [0, 0, 0]
