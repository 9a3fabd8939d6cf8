"""indexer_topk on the GPU against the oracle (bit-exact index lists), and the index lists it
writes feeding sparse_mla_decode on the same stream."""
import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import attention, pack, topk
from tests.gpu_util import assert_close, bf16_dev, i32

pytestmark = pytest.mark.gpu


def _run(logits, L, Q, K):
    out = m.indexer_topk(torch.from_numpy(logits).cuda(), i32(L), K)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("B,Q,S,K", [(3, 1, 1000, 64), (2, 4, 20000, 2048), (4, 2, 9000, 100), (1, 1, 64, 2048),
                                     (2, 3, 40000, 8192), (5, 1, 8, 3), (2, 16, 6000, 300), (1, 16, 30000, 8192)])
def test_random_rows_with_ties_nan_and_signed_zero(B, Q, S, K):
    rng = np.random.default_rng(B * 1000 + S)
    logits = rng.standard_normal((B, Q, S)).astype(np.float32)
    logits[0] = np.round(logits[0] * 4) / 4                      # many ties
    flat = logits.reshape(-1)
    flat[rng.integers(0, flat.size, size=max(1, flat.size // 200))] = np.nan
    flat[rng.integers(0, flat.size, size=max(1, flat.size // 200))] = -0.0
    flat[rng.integers(0, flat.size, size=max(1, flat.size // 200))] = 0.0
    flat[rng.integers(0, flat.size, size=max(1, flat.size // 500))] = np.inf
    flat[rng.integers(0, flat.size, size=max(1, flat.size // 500))] = -np.inf
    bits = flat.view(np.uint32)                                     # NaNs with the sign set and with payloads
    for pattern in (0xFFC00000, 0xFF800001, 0xFFFFFFFF, 0x7F800001, 0x7FFFFFFF):
        bits[rng.integers(0, flat.size, size=max(1, flat.size // 1000))] = pattern
    L = rng.integers(1, S + Q + 3, size=B).astype(np.int32)      # some ranges exceed the row (capped)
    L[0] = S + Q - 1                                               # the full row for the last query
    np.testing.assert_array_equal(_run(logits, L, Q, K), topk.select(logits, L, Q, K))


@pytest.mark.parametrize("B,Q", [(20, 1), (40, 1), (100, 2)], ids=["7-CTA clusters", "3-CTA clusters", "one CTA per row"])
def test_row_counts_that_change_the_launch(B, Q):
    """The launch splits a row over SMs // rows CTAs (2..8) when the batch leaves SMs idle and uses
    one CTA per row otherwise: 20 and 40 rows give clusters of 7 and 3 CTAs on 152 SMs, 200 rows
    one CTA each. Rows of uneven length and ties in one request."""
    rng = np.random.default_rng(B * 7 + Q)
    S, K = 9000, 700
    logits = rng.standard_normal((B, Q, S)).astype(np.float32)
    logits[1] = np.round(logits[1] * 2) / 2
    L = rng.integers(500, S + Q, size=B).astype(np.int32)
    np.testing.assert_array_equal(_run(logits, L, Q, K), topk.select(logits, L, Q, K))


@pytest.mark.parametrize("S", [5000, 20000])      # 20,000 equal keys overflow the candidate store
def test_degenerate_rows(S):
    K = 2048
    mixed = np.full(S, -np.inf, np.float32)
    mixed.view(np.uint32)[::3] = 0xFF800001                         # negative NaN
    mixed.view(np.uint32)[1::3] = 0x7FC00000                        # positive NaN
    mixed[::97] = -1.0
    logits = np.stack([np.full(S, 1.5, np.float32), np.full(S, np.nan, np.float32), mixed,
                       np.arange(S, dtype=np.float32)[::-1].copy(), -np.arange(S, dtype=np.float32)])[:, None]
    L = np.array([S, S, S, S, 1000], np.int32)
    np.testing.assert_array_equal(_run(logits, L, 1, K), topk.select(logits, L, 1, K))


def test_sample_that_misleads_the_bound():
    """The sampled positions (8 in every 128) hold the largest logits, spread over several bins,
    so a bound taken from the sample leaves fewer than K keys above it and the select must fall
    back; a second row has its K-th key in a bin of more than 8,192 ties."""
    rng = np.random.default_rng(11)
    S, K = 40000, 2048
    logits = rng.standard_normal((2, 1, S)).astype(np.float32)
    sampled = (np.arange(S) >> 3) % 16 == 0
    logits[0, 0, sampled] = 10 + 5 * rng.random(int(sampled.sum()), dtype=np.float32)
    logits[1, 0, :12000] = 3.0
    L = np.array([S, S], np.int32)
    np.testing.assert_array_equal(_run(logits, L, 1, K), topk.select(logits, L, 1, K))


def test_rows_longer_than_the_bitmap():
    """Rows past 262,144 positions take the general path; one row stays just inside."""
    rng = np.random.default_rng(9)
    S = 300_000
    logits = rng.standard_normal((3, 1, S)).astype(np.float32)
    logits[1, 0] = np.round(logits[1, 0] * 8) / 8
    L = np.array([S, 262_144, 270_000], np.int32)
    np.testing.assert_array_equal(_run(logits, L, 1, 2048), topk.select(logits, L, 1, 2048))


def test_headline_shape_is_exact():
    """B=64 query tokens, ranges uniform in [70K, 160K], K = 2,048, as in the decode workload."""
    case = workloads.make_case(2)
    S = int(case.seq_lens.max())
    S = (S + 3) // 4 * 4
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((case.B, 1, S)).astype(np.float32)
    np.testing.assert_array_equal(_run(logits, case.seq_lens, 1, case.topk),
                                  topk.select(logits, case.seq_lens, 1, case.topk))


def test_topk_feeds_decode_on_one_stream():
    case = workloads.small_case(B=3, Q=2, H=32, topk=512, L=(3000, 900, 2200), seed=61)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    rows = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    S = 3000
    logits = np.random.default_rng(62).standard_normal((case.B, case.Q, S)).astype(np.float32)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        cache = torch.zeros((case.num_pages, 64, 352), dtype=torch.uint8, device="cuda")
        m.mla_kv_pack(bf16_dev(lat), bf16_dev(rope), torch.arange(case.num_pages * 64, device="cuda"), cache,
                      stream=stream)
        sl = i32(case.seq_lens)
        idx = m.indexer_topk(torch.from_numpy(logits).cuda(), sl, case.topk, stream=stream)
        out, lse = m.sparse_mla_decode(bf16_dev(case.q_bits), cache, i32(case.page_table), idx, sl,
                                       case.softmax_scale, stream=stream)
    torch.cuda.synchronize()
    ref_idx = topk.select(logits, case.seq_lens, case.Q, case.topk)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    ref_out, ref_lse = attention.sparse_decode(case.q_bits, rows, case.page_table, ref_idx, case.seq_lens,
                                               case.softmax_scale)
    assert_close(out, lse, ref_out, ref_lse, "indexer_topk -> sparse_mla_decode")


def test_rejects_bad_arguments_before_launch():
    import ctypes
    lib = m.load_library()
    V = ctypes.c_void_p
    x = torch.arange(64, dtype=torch.float32, device="cuda").reshape(1, 1, 64)
    sl = torch.full((1,), 64, dtype=torch.int32, device="cuda")
    out = torch.full((1, 1, 8), 7, dtype=torch.int32, device="cuda")
    P = lambda t: V(t.data_ptr())
    assert lib.indexer_topk(P(x), 64, P(sl), 1, 1, 8, P(out), None) == 0
    assert lib.indexer_topk(P(x), 62, P(sl), 1, 1, 8, P(out), None) == 2          # stride not a multiple of 4
    assert lib.indexer_topk(V(x.data_ptr() + 4), 64, P(sl), 1, 1, 8, P(out), None) == 2
    assert lib.indexer_topk(P(x), 64, P(sl), 1, 1, 0, P(out), None) == 1
    assert lib.indexer_topk(P(x), 64, P(sl), 1, 17, 8, P(out), None) == 1
    host = torch.zeros((1, 1, 64), dtype=torch.float32)
    assert lib.indexer_topk(P(host), 64, P(sl), 1, 1, 8, P(out), None) == 1       # host memory
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [[[56, 57, 58, 59, 60, 61, 62, 63]]]            # only the first call ran
