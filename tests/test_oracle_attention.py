"""Pins for the oracle's dequantisation and sparse / dense decode (CPU only).

Checked against: torch's scaled_dot_product_attention in float64 (a library
routine), closed forms for one and two tokens, a pure-Python brute force on
tiny inputs that enumerates masked entries, and invariants (softmax mass 1,
top-k = all equals dense, index and page permutation).
"""
import itertools
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention, codec, pack


def _cache_for(case, fill=None):
    cache = np.zeros((case.num_pages, 64, 352), np.uint8)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    cache[:] = pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352)
    return cache


def test_dequant_known_bytes():
    row = np.zeros((1, 352), np.uint8)
    row[0, 0] = 0x7 | (0xF << 4)      # +6, -6
    row[0, 1] = 0x1 | (0x9 << 4)      # +0.5, -0.5
    row[0, 256] = 0x38                # scale 1.0 for block 0
    row[0, 257] = 0x01                # scale 2^-9 for block 1
    row[0, 8] = 0x5                   # element 16 (block 1): +3
    row[0, 288] = 0x38                # rope[0] = 1.0
    row[0, 289] = 0xFE                # rope[1] = -448
    row[0, 290] = 0x01                # rope[2] = 2^-9
    c = attention.dequant_rows(row)[0]
    assert c[:4].tolist() == [6.0, -6.0, 0.5, -0.5]
    assert c[16] == 3.0 * 2.0 ** -9
    assert c[512:515].tolist() == [1.0, -448.0, 2.0 ** -9]


def test_matches_torch_sdpa_fp64():
    case = workloads.small_case(B=2, Q=2, H=4, topk=150, L=(500, 900), seed=11)
    cache = _cache_for(case)
    out, lse = attention.sparse_decode(case.q_bits, cache, case.page_table, case.topk_indices,
                                       case.seq_lens, case.softmax_scale)
    q = codec.bf16_bits_to_f64(case.q_bits)
    for b in range(case.B):
        for j in range(case.Q):
            idx = case.topk_indices[b, j].astype(np.int64)
            pg = case.page_table[b][idx // 64]
            c = attention.dequant_rows(cache[pg, idx % 64])
            qt = torch.from_numpy(q[b, j])[None, :, None, :]          # [1, H, 1, 576]
            kt = torch.from_numpy(c)[None, None].expand(1, case.H, -1, -1)
            vt = torch.from_numpy(c[:, :512])[None, None].expand(1, case.H, -1, -1)
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=case.softmax_scale)
            np.testing.assert_allclose(out[b, j], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)
            z = case.softmax_scale * (torch.from_numpy(q[b, j]) @ torch.from_numpy(c).T)
            np.testing.assert_allclose(lse[b, j], torch.logsumexp(z, dim=1).numpy(), rtol=1e-13, atol=1e-13)


def test_softmax_mass_is_one():
    case = workloads.small_case(B=1, Q=1, H=8, topk=300, L=(2000,), seed=5)
    cache = _cache_for(case)
    _, lse = attention.sparse_decode(case.q_bits, cache, case.page_table, case.topk_indices,
                                     case.seq_lens, case.softmax_scale)
    q = codec.bf16_bits_to_f64(case.q_bits)[0, 0]
    idx = case.topk_indices[0, 0]
    c = attention.dequant_rows(cache[case.page_table[0][idx // 64], idx % 64])
    z = case.softmax_scale * (q @ c.T)
    mass = np.exp(z - lse[0, 0][:, None]).sum(axis=1)
    np.testing.assert_allclose(mass, 1.0, rtol=0, atol=1e-12)


def test_sparse_with_all_positions_equals_dense():
    case = workloads.small_case(B=2, Q=1, H=4, topk=10, L=(300, 190), seed=9)
    cache = _cache_for(case)
    K = int(case.seq_lens.max())
    topk = -np.ones((case.B, 1, K), np.int32)
    for b in range(case.B):
        topk[b, 0, :case.seq_lens[b]] = np.random.default_rng(b).permutation(case.seq_lens[b])
    out_s, lse_s = attention.sparse_decode(case.q_bits, cache, case.page_table, topk, case.seq_lens,
                                           case.softmax_scale)
    out_d, lse_d = attention.dense_decode(case.q_bits, cache, case.page_table, case.seq_lens,
                                          case.softmax_scale)
    np.testing.assert_allclose(out_s, out_d, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse_s, lse_d, rtol=1e-13, atol=1e-13)


def _one_query_case(H, idx, L, num_pages=3, seed=1):
    case = workloads.small_case(B=1, Q=1, H=H, topk=len(idx), L=(L,), num_pages=num_pages, seed=seed)
    case.topk_indices = np.array(idx, np.int32).reshape(1, 1, -1)
    return case


def test_single_valid_token_closed_form():
    case = _one_query_case(4, [37, -1, -1], 100)
    cache = _cache_for(case)
    out, lse = attention.sparse_decode(case.q_bits, cache, case.page_table, case.topk_indices,
                                       case.seq_lens, case.softmax_scale)
    c = attention.dequant_rows(cache[case.page_table[0][0], 37][None])[0]
    q = codec.bf16_bits_to_f64(case.q_bits)[0, 0]
    np.testing.assert_array_equal(out[0, 0], np.broadcast_to(c[:512], (4, 512)))
    np.testing.assert_allclose(lse[0, 0], case.softmax_scale * (q @ c), rtol=1e-14)


def test_two_tokens_closed_form():
    case = _one_query_case(3, [3, 70], 100)
    cache = _cache_for(case)
    out, lse = attention.sparse_decode(case.q_bits, cache, case.page_table, case.topk_indices,
                                       case.seq_lens, case.softmax_scale)
    c1 = attention.dequant_rows(cache[case.page_table[0][0], 3][None])[0]
    c2 = attention.dequant_rows(cache[case.page_table[0][1], 70 % 64][None])[0]
    q = codec.bf16_bits_to_f64(case.q_bits)[0, 0]
    for h in range(3):
        z1, z2 = case.softmax_scale * (q[h] @ c1), case.softmax_scale * (q[h] @ c2)
        w1 = 1.0 / (1.0 + math.exp(z2 - z1))
        np.testing.assert_allclose(out[0, 0, h], w1 * c1[:512] + (1 - w1) * c2[:512], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[0, 0, h], max(z1, z2) + math.log1p(math.exp(-abs(z1 - z2))), rtol=1e-13)


def test_bruteforce_tiny_with_every_mask_kind():
    """H=1, Q=2, up to 4 entries drawn from a pool that holds valid positions,
    -1, other negatives, positions past seq_len, a position past the first
    query's causal limit, and positions whose page-table entry is bad."""
    L = 130          # pages 0..2 used; position 129 is the last token
    pool = [0, 5, 64, 128, 129, -1, -7, 130, 200, 191]
    base = workloads.small_case(B=1, Q=2, H=1, topk=4, L=(L,), num_pages=4, seed=21)
    cache = _cache_for(base)
    page_row = base.page_table[0].copy()
    page_row = np.concatenate([page_row, [-1, 99]]).astype(np.int32)   # cols 3, 4: bad entries
    table = page_row[None]
    q = codec.bf16_bits_to_f64(base.q_bits)
    n_checked = 0
    for n in range(0, 5):
        for combo in itertools.islice(itertools.combinations_with_replacement(pool, n), 0, None, 7):
            idx = np.array(list(combo) + [-1] * (4 - n), np.int32)
            topk = np.stack([idx, idx])[None]
            out, lse = attention.sparse_decode(base.q_bits, cache, table, topk, base.seq_lens, base.softmax_scale)
            for j in range(2):
                causal = L - 2 + j
                zs, vs = [], []
                for t in idx.tolist():
                    if t < 0 or t >= L or t > causal:
                        continue
                    col = t // 64
                    pg = int(table[0][col]) if col < table.shape[1] else -1
                    if pg < 0 or pg >= base.num_pages:
                        continue
                    c = attention.dequant_rows(cache[pg, t % 64][None])[0]
                    zs.append(base.softmax_scale * sum(q[0, j, 0, d] * c[d] for d in range(576)))
                    vs.append(c[:512])
                if not zs:
                    assert (out[0, j] == 0).all() and np.isneginf(lse[0, j]).all()
                    continue
                m = max(zs)
                w = [math.exp(z - m) for z in zs]
                s = sum(w)
                ref = sum(wi * v for wi, v in zip(w, vs)) / s
                np.testing.assert_allclose(out[0, j, 0], ref, rtol=1e-12, atol=1e-12)
                assert abs(lse[0, j, 0] - (m + math.log(s))) < 1e-12
                n_checked += 1
    assert n_checked > 40


def test_index_and_page_permutation_invariance():
    case = workloads.small_case(B=2, Q=1, H=4, topk=180, L=(700, 333), seed=13)
    cache = _cache_for(case)
    out, lse = attention.sparse_decode(case.q_bits, cache, case.page_table, case.topk_indices,
                                       case.seq_lens, case.softmax_scale)
    rng = np.random.default_rng(0)
    topk2 = case.topk_indices.copy()
    for b in range(case.B):
        topk2[b, 0] = rng.permutation(topk2[b, 0])
    out2, lse2 = attention.sparse_decode(case.q_bits, cache, case.page_table, topk2, case.seq_lens,
                                         case.softmax_scale)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-13)
    # physical page permutation with the page table updated: identical result
    perm = rng.permutation(case.num_pages)
    cache3 = np.empty_like(cache)
    cache3[perm] = cache
    table3 = np.where(case.page_table >= 0, perm[np.clip(case.page_table, 0, None)], -1).astype(np.int32)
    out3, lse3 = attention.sparse_decode(case.q_bits, cache3, table3, case.topk_indices, case.seq_lens,
                                         case.softmax_scale)
    np.testing.assert_array_equal(out3, out)
    np.testing.assert_array_equal(lse3, lse)


def test_duplicates_count_twice():
    case = _one_query_case(2, [10, 10, 50], 100)
    cache = _cache_for(case)
    out, lse = attention.sparse_decode(case.q_bits, cache, case.page_table, case.topk_indices,
                                       case.seq_lens, case.softmax_scale)
    c1 = attention.dequant_rows(cache[case.page_table[0][0], 10][None])[0]
    c2 = attention.dequant_rows(cache[case.page_table[0][0], 50][None])[0]
    q = codec.bf16_bits_to_f64(case.q_bits)[0, 0]
    for h in range(2):
        z1, z2 = case.softmax_scale * (q[h] @ c1), case.softmax_scale * (q[h] @ c2)
        w1 = 2 * math.exp(z1) / (2 * math.exp(z1) + math.exp(z2))
        np.testing.assert_allclose(out[0, 0, h], w1 * c1[:512] + (1 - w1) * c2[:512], rtol=1e-12, atol=1e-12)
