"""The FP8 comparison paths on the GPU against the oracle: the FP8 and per-token FP8 row packs and
the staging kernel bit-exact, the FP8 decodes and the staged path within the decode tolerance (the
reference is fp64 attention over the same rows)."""
import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import codec, fp8rows, pack
from tests.gpu_util import assert_close, bf16_dev, decode_inputs, i32, oracle_units_from_device_rows

pytestmark = pytest.mark.gpu


def _bf16_rows(n, seed, special=False):
    rng = np.random.default_rng(seed)
    lat = (rng.standard_normal((n, 512)) * rng.lognormal(0, 1.5, (n, 1)) * 40).astype(np.float32)
    rope = (rng.standard_normal((n, 64)) * 3).astype(np.float32)
    if special:
        lat[0, :6] = [np.nan, -np.nan, np.inf, -np.inf, -0.0, 1e-30]
        rope[1, :4] = [np.nan, -np.inf, 500.0, -0.0]
        lat[2] = 0.0
        lat[3, 100:116] = 448.0 * np.array([1, 1.0625, 1.0626, 2, 1e3, -1e5, 0.5, 1 / 3] * 2, np.float32)
    return workloads.f32_to_bf16_bits(lat), workloads.f32_to_bf16_bits(rope)


def test_fp8_pack_bit_exact_with_slot_rules():
    lat, rope = _bf16_rows(700, 1, special=True)
    pages = 12
    slots = np.arange(700, dtype=np.int64)
    slots[5] = -1
    slots[6] = pages * 64 + 3            # outside: skipped and counted
    slots[7] = -5                        # negative other than -1: skipped and counted
    cache = torch.zeros((pages, 64, 576), dtype=torch.uint8, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    m.fp8_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.from_numpy(slots).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    ref = np.zeros((pages, 64, 576), np.uint8)
    fp8rows.write_cache_fp8(ref, lat, rope, slots)
    np.testing.assert_array_equal(cache.cpu().numpy(), ref)
    assert status.cpu().tolist() == [0, 0, 0, 2]


def test_stage_bit_exact():
    case = workloads.small_case(B=3, Q=2, H=16, topk=192, L=(500, 700, 64), invalid_frac=0.2, dup=True,
                                causal_tail=True, seed=5)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope)
    rows[7, 256] = 0x7F                                  # a NaN scale byte (pack never writes one)
    rows = rows.reshape(case.num_pages, 64, 352)
    cache = torch.from_numpy(rows.copy()).cuda()
    _, pt, tk, sl = decode_inputs(case)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    staged, sidx, spt, ssl = m.nvfp4_stage_fp8(cache, pt, tk, sl, dev_status=status)
    torch.cuda.synchronize()
    ref_rows, written, ref_idx, ref_pt, ref_sl = fp8rows.stage(rows, case.page_table, case.topk_indices,
                                                               case.seq_lens, case.Q)
    got = staged.cpu().numpy().reshape(-1, 576)
    np.testing.assert_array_equal(got[written], ref_rows[written])
    np.testing.assert_array_equal(sidx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(spt.cpu().numpy(), ref_pt)
    np.testing.assert_array_equal(ssl.cpu().numpy(), ref_sl)
    # the entries the decode would count as bad are counted the same way
    dstat = torch.zeros(4, dtype=torch.int32, device="cuda")
    q, pt2, tk2, sl2 = decode_inputs(case)
    m.sparse_mla_decode(q, cache, pt2, tk2, sl2, case.softmax_scale, dev_status=dstat)
    torch.cuda.synchronize()
    assert status.cpu().tolist()[:2] == dstat.cpu().tolist()[:2]


SMALL = [
    dict(B=2, Q=1, H=16, topk=200, L=(700, 1000)),
    dict(B=1, Q=4, H=32, topk=256, L=(3000,)),
    dict(B=3, Q=2, H=64, topk=130, L=(500, 600, 700)),
    dict(B=2, Q=2, H=32, topk=384, L=(1500, 1400), invalid_frac=0.25, dup=True, causal_tail=True),
    dict(B=4, Q=1, H=16, topk=50, L=(40, 60, 2000, 64)),
]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: "B{B}Q{Q}H{H}K{topk}".format(**s))
def test_fp8_decode_matches_oracle(spec):
    case = workloads.small_case(seed=40 + len(str(spec)), **spec)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    n = case.num_pages * 64
    cache = torch.zeros((case.num_pages, 64, 576), dtype=torch.uint8, device="cuda")
    m.fp8_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(n, device="cuda"), cache)
    q, pt, tk, sl = decode_inputs(case)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = m.sparse_mla_decode_fp8(q, cache, pt, tk, sl, case.softmax_scale, dev_status=status)
    torch.cuda.synchronize()
    ref_cache = np.zeros((case.num_pages, 64, 576), np.uint8)
    fp8rows.write_cache_fp8(ref_cache, lat, rope, np.arange(n))
    np.testing.assert_array_equal(cache.cpu().numpy(), ref_cache)
    ref_out, ref_lse = fp8rows.sparse_decode_fp8(case.q_bits, ref_cache, case.page_table, case.topk_indices,
                                                 case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, f"fp8 {spec}")
    assert status.cpu().tolist()[2] == 0


@pytest.mark.parametrize("spec", SMALL[:4], ids=lambda s: "B{B}Q{Q}H{H}K{topk}".format(**s))
def test_staged_path_matches_oracle(spec):
    spec = dict(spec, topk=(spec["topk"] + 63) // 64 * 64)          # the staged path takes whole 64-row pages
    case = workloads.small_case(seed=60 + len(str(spec)), **spec)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    cache = torch.from_numpy(rows.copy()).cuda()
    q, pt, tk, sl = decode_inputs(case)
    out, lse, _ = m.staged_sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale)
    torch.cuda.synchronize()
    staged, _, sidx, spt, ssl = fp8rows.stage(rows, case.page_table, case.topk_indices, case.seq_lens, case.Q)
    qs = case.q_bits.reshape(case.B * case.Q, 1, case.H, 576)
    ref_out, ref_lse = fp8rows.sparse_decode_fp8(qs, staged.reshape(-1, 64, 576), spt, sidx, ssl,
                                                 case.softmax_scale)
    assert_close(out, lse, ref_out.reshape(out.shape), ref_lse.reshape(lse.shape), f"staged {spec}")


def test_token_pack_bit_exact_with_slot_rules():
    lat, rope = _bf16_rows(700, 2)
    lat[5] = 0                                          # an all-zero latent: the scale comes from the 1e-26 floor
    pages = 12
    slots = np.arange(700, dtype=np.int64)
    slots[9] = -1
    slots[10] = pages * 64 + 7
    cache = torch.full((pages, 64, 672), 0xAB, dtype=torch.uint8, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    m.fp8_token_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.from_numpy(slots).cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    ref = np.full((pages, 64, 672), 0xAB, np.uint8)
    fp8rows.write_cache_token(ref, lat, rope, slots)
    np.testing.assert_array_equal(cache.cpu().numpy(), ref)
    assert status.cpu().tolist() == [0, 0, 0, 1]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: "B{B}Q{Q}H{H}K{topk}".format(**s))
def test_token_decode_matches_oracle(spec):
    case = workloads.small_case(seed=80 + len(str(spec)), **spec)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    n = case.num_pages * 64
    cache = torch.zeros((case.num_pages, 64, 672), dtype=torch.uint8, device="cuda")
    m.fp8_token_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(n, device="cuda"), cache)
    q, pt, tk, sl = decode_inputs(case)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out, lse = m.sparse_mla_decode_fp8_token(q, cache, pt, tk, sl, case.softmax_scale, dev_status=status)
    torch.cuda.synchronize()
    ref_cache = np.zeros((case.num_pages, 64, 672), np.uint8)
    fp8rows.write_cache_token(ref_cache, lat, rope, np.arange(n))
    np.testing.assert_array_equal(cache.cpu().numpy(), ref_cache)
    ref_out, ref_lse = fp8rows.sparse_decode_token(case.q_bits, ref_cache, case.page_table, case.topk_indices,
                                                   case.seq_lens, case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, f"per-token {spec}")
    assert status.cpu().tolist()[2] == 0


@pytest.mark.parametrize("path", ["fp8", "staged", "token"])
def test_headline_size_sampled_units(path):
    """The 64-query headline workload through either comparison path, with the launch
    configuration the bench times; 8 query tokens checked against the oracle on their own rows."""
    case = workloads.make_case(2)
    n = case.num_pages * 64
    lat, rope = workloads.device_rows(case, n, "cuda")
    q, pt, tk, sl = decode_inputs(case)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    if path == "fp8":
        cache = torch.empty((case.num_pages, 64, 576), dtype=torch.uint8, device="cuda")
        m.fp8_kv_pack(lat, rope, torch.arange(n, device="cuda"), cache)
        out, lse = m.sparse_mla_decode_fp8(q, cache, pt, tk, sl, case.softmax_scale, dev_status=status)
    elif path == "token":
        cache = torch.empty((case.num_pages, 64, 672), dtype=torch.uint8, device="cuda")
        m.fp8_token_kv_pack(lat, rope, torch.arange(n, device="cuda"), cache)
        out, lse = m.sparse_mla_decode_fp8_token(q, cache, pt, tk, sl, case.softmax_scale, dev_status=status)
    else:
        cache = torch.empty((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
        m.mla_kv_pack(lat, rope, torch.arange(n, device="cuda"), cache)
        out, lse, _ = m.staged_sparse_mla_decode(q, cache, pt, tk, sl, case.softmax_scale, dev_status=status)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    units = [(b, 0) for b in (0, 1, 17, 31, 32, 45, 62, 63)]
    ref = oracle_units_from_device_rows(case, units, lat, rope, fmt=path)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for (b, j), (ro, rl) in ref.items():
        assert_close(o[b, j], l[b, j], ro, rl, f"{path} unit {(b, j)}")
    assert np.isfinite(o).all()


def test_fp8_decode_rejects_host_results():
    case = workloads.small_case(B=1, Q=1, H=16, topk=64, L=(200,), seed=3)
    q, pt, tk, sl = decode_inputs(case)
    cache = torch.zeros((case.num_pages, 64, 576), dtype=torch.uint8, device="cuda")
    hout = torch.empty((1, 1, 16, 512), dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((1, 1, 16), dtype=torch.float32).pin_memory()
    lib = m.load_library()
    ws = torch.empty(m.sparse_mla_decode_workspace_size(1, 1, 16, 64), dtype=torch.uint8, device="cuda")
    P = lambda t: None if t is None else __import__("ctypes").c_void_p(t.data_ptr())
    rc = lib.sparse_mla_decode_fp8(P(q), P(cache), case.num_pages, P(pt), pt.shape[1], P(tk), P(sl), 1, 1, 16, 64,
                                   case.softmax_scale, P(hout), P(hlse), P(ws), ws.numel(), None, None)
    assert rc == 3   # NVFP4MLA_ERR_UNSUPPORTED
