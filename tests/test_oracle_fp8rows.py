"""Pins for the oracle's FP8 576-byte rows and staged copy (CPU only).

Checked against: torch's float8_e4m3fn conversion (a library round-to-nearest-even) for every
rounding, the row layout spelled out byte by byte, a per-entry brute force of the staging
(validity rule, page lookup, destination row), and torch's scaled_dot_product_attention in
float64 for the decode over FP8 rows.
"""
import numpy as np
import torch

import workloads
from oracle import attention, codec, fp8rows, pack


def _torch_e4m3(x):
    """torch's E4M3 bytes of float64 values below 464 in magnitude (torch makes larger ones NaN)."""
    return torch.from_numpy(np.asarray(x, np.float64).astype(np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_fp8_row_layout_and_rounding():
    rng = np.random.default_rng(0)
    lat = workloads.f32_to_bf16_bits((rng.standard_normal((50, 512)) * 30).astype(np.float32))
    rope = workloads.f32_to_bf16_bits((rng.standard_normal((50, 64)) * 3).astype(np.float32))
    rows = fp8rows.encode_rows_fp8(lat, rope)
    assert rows.shape == (50, 576) and rows.dtype == np.uint8
    xl, xr = codec.bf16_bits_to_f64(lat), codec.bf16_bits_to_f64(rope)
    m = np.abs(xl) < 464
    np.testing.assert_array_equal(rows[:, :512][m], _torch_e4m3(xl[m]))
    np.testing.assert_array_equal(rows[:, :512][~m] & 0x7F, 0x7E)                     # saturated at 448
    np.testing.assert_array_equal(rows[:, 512:], _torch_e4m3(xr))
    # the rope bytes are the same bytes the NVFP4 row carries
    np.testing.assert_array_equal(rows[:, 512:], pack.encode_rows(lat, rope)[:, 288:352])
    np.testing.assert_array_equal(fp8rows.dequant_rows_fp8(rows),
                                  torch.from_numpy(rows).view(torch.float8_e4m3fn).to(torch.float64).numpy())


def test_staged_copy_rounds_the_dequantised_value_once():
    rng = np.random.default_rng(1)
    rows = rng.integers(0, 256, size=(200, 352), dtype=np.uint8)
    rows[:, 256:288] = rng.integers(0, 0x7F, size=(200, 32))          # finite scales of either sign bit off
    rows[:3, 256:288] = 0x7E                                           # scale 448: values up to 6 * 448
    staged = fp8rows.stage_rows(rows)
    assert staged.shape == (200, 576)
    # latent: independent decode of the nibbles and scales, rounded by torch
    nib = rows[:, :256].astype(np.int64)
    codes = np.stack([nib & 15, nib >> 4], axis=2).reshape(200, 512)
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    val = np.where(codes & 8, -1.0, 1.0) * e2m1[codes & 7]
    scl = torch.from_numpy(rows[:, 256:288].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    val = val * np.repeat(scl, 16, axis=1)
    small = np.abs(val) < 464
    np.testing.assert_array_equal(staged[:, :512][small], _torch_e4m3(val[small]))
    assert (~small).any()
    np.testing.assert_array_equal(staged[:, :512][~small] & 0x7F, 0x7E)
    np.testing.assert_array_equal(staged[:, :512][~small] >> 7, (val[~small] < 0).astype(np.uint8))
    np.testing.assert_array_equal(staged[:, 512:], rows[:, 288:352])
    # a NaN scale byte (never written by pack) stages its block as 0x7F
    odd = rows[:2].copy()
    odd[0, 256] = 0x7F
    odd[1, 257] = 0xFF
    st = fp8rows.stage_rows(odd)
    assert (st[0, :16] == 0x7F).all() and (st[1, 16:32] == 0x7F).all()
    np.testing.assert_array_equal(st[0, 16:], staged[0, 16:])
    # the staged value is the E4M3 value nearest the dequantised one: never off by more than half a step
    got = fp8rows.dequant_rows_fp8(staged)[:, :512]
    assert np.all(np.abs(got[small] - val[small]) <= np.maximum(np.abs(val[small]) / 16, 2.0 ** -10))


def _small_case_cache(**kw):
    case = workloads.small_case(**kw)
    lat, rope = workloads.host_rows(case, np.arange(case.num_pages))
    return case, pack.encode_rows(lat, rope).reshape(case.num_pages, 64, 352), lat, rope


def test_stage_brute_force():
    case, cache, _, _ = _small_case_cache(B=3, Q=2, H=16, topk=192, L=(500, 700, 64), invalid_frac=0.2,
                                          dup=True, causal_tail=True, seed=5)
    staged, written, tk, pt, sl = fp8rows.stage(cache, case.page_table, case.topk_indices, case.seq_lens, case.Q)
    K = case.topk
    assert tk.shape == (case.B * case.Q, 1, K) and pt.shape == (case.B * case.Q, K // 64)
    assert (sl == K).all()
    n_used = 0
    for b in range(case.B):
        L = int(case.seq_lens[b])
        for j in range(case.Q):
            u = b * case.Q + j
            for i, e in enumerate(case.topk_indices[b, j].tolist()):
                usable = 0 <= e < L and e <= L - case.Q + j and e // 64 < case.page_table.shape[1]
                page = int(case.page_table[b, e // 64]) if usable else -1
                usable = usable and 0 <= page < case.num_pages
                assert written[u * K + i] == usable and tk[u, 0, i] == (i if usable else -1)
                if usable:
                    n_used += 1
                    np.testing.assert_array_equal(staged[u * K + i],
                                                  fp8rows.stage_rows(cache[page, e % 64][None])[0])
                    # the identity page table reaches exactly this staged row
                    assert pt[u, i // 64] * 64 + i % 64 == u * K + i
                else:
                    assert not staged[u * K + i].any()
    assert 0 < n_used < case.B * case.Q * K


def test_fp8_decode_matches_torch_sdpa_and_the_staged_pipeline():
    case, cache, lat, rope = _small_case_cache(B=2, Q=2, H=4, topk=128, L=(500, 900), seed=12)
    cache8 = np.zeros((case.num_pages, 64, 576), np.uint8)
    fp8rows.write_cache_fp8(cache8, lat, rope, np.arange(case.num_pages * 64))
    out, lse = fp8rows.sparse_decode_fp8(case.q_bits, cache8, case.page_table, case.topk_indices,
                                         case.seq_lens, case.softmax_scale)
    q = codec.bf16_bits_to_f64(case.q_bits)
    for b in range(case.B):
        for j in range(case.Q):
            idx = case.topk_indices[b, j].astype(np.int64)
            pg = case.page_table[b][idx // 64]
            c = torch.from_numpy(cache8[pg, idx % 64].copy()).view(torch.float8_e4m3fn).to(torch.float64)
            qt = torch.from_numpy(q[b, j])[None, :, None, :]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, c[None, None].expand(1, case.H, -1, -1), c[None, None, :, :512].expand(1, case.H, -1, -1),
                scale=case.softmax_scale)
            np.testing.assert_allclose(out[b, j], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)
    # staged pipeline: the FP8 decode over the staged rows as B*Q one-query requests equals attention
    # over the staged copies of each query's usable rows, and stays close to the NVFP4 result
    staged, _, tk, pt, sl = fp8rows.stage(cache, case.page_table, case.topk_indices, case.seq_lens, case.Q)
    qs = case.q_bits.reshape(case.B * case.Q, 1, case.H, 576)
    so, sls = fp8rows.sparse_decode_fp8(qs, staged.reshape(-1, 64, 576), pt, tk, sl, case.softmax_scale)
    no, nls = attention.sparse_decode(case.q_bits, cache, case.page_table, case.topk_indices, case.seq_lens,
                                      case.softmax_scale)
    for b in range(case.B):
        for j in range(case.Q):
            u = b * case.Q + j
            idx = case.topk_indices[b, j].astype(np.int64)
            ok = attention.valid_entries(idx, int(case.seq_lens[b]), int(case.seq_lens[b]) - case.Q + j,
                                         case.page_table[b], case.num_pages)
            rows = cache[case.page_table[b][idx[ok] // 64], idx[ok] % 64]
            o, l = attention.attend(q[b, j], fp8rows.dequant_rows_fp8(fp8rows.stage_rows(rows)), case.softmax_scale)
            np.testing.assert_allclose(so[u, 0], o, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(sls[u, 0], l, rtol=1e-13, atol=1e-13)
    assert np.max(np.abs(so.reshape(no.shape) - no)) < 0.1 * np.max(np.abs(no))


def test_per_token_rows_against_torch_roundings_and_bounds():
    """Per-token FP8 rows: fp32 scale and divisions, then torch's E4M3 and bf16 conversions (library
    roundings) on the same fp32 quotients; the latent's largest element codes as 448; the
    dequantised latent is within half an E4M3 step of the input; the layout byte by byte."""
    rng = np.random.default_rng(7)
    n = 64
    lat32 = (rng.standard_normal((n, 512)) * rng.lognormal(0, 2, (n, 1))).astype(np.float32)
    lat32[0] = 0.0                                                     # all-zero row: scale from the 1e-26 floor
    lat = workloads.f32_to_bf16_bits(lat32)
    rope = workloads.f32_to_bf16_bits((rng.standard_normal((n, 64)) * 2).astype(np.float32))
    rows = fp8rows.encode_rows_token(lat, rope)
    assert rows.shape == (n, 672) and not rows[:, 644:].any()
    x = torch.from_numpy(codec.bf16_bits_to_f64(lat)).float()
    r = torch.from_numpy(codec.bf16_bits_to_f64(rope)).float()
    scale = torch.clamp(x.abs().amax(dim=1, keepdim=True), min=1e-26) / 448.0
    np.testing.assert_array_equal(rows[:, 640:644].copy().view("<f4"), scale.numpy())
    np.testing.assert_array_equal(rows[:, :512], (x / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    np.testing.assert_array_equal(rows[:, 512:640].copy().view("<u2"),
                                  (r / scale).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    big = np.abs(codec.bf16_bits_to_f64(lat)).argmax(axis=1)
    assert all((rows[i, big[i]] & 0x7F) == 0x7E for i in range(1, n))           # amax -> 448
    d = fp8rows.dequant_rows_token(rows)
    xl = codec.bf16_bits_to_f64(lat)
    s = rows[:, 640:644].copy().view("<f4").astype(np.float64)
    assert np.all(np.abs(d[:, :512] - xl) <= np.maximum(np.abs(xl) / 16, s * 2.0 ** -10) * (1 + 1e-6))
    assert np.all(np.abs(d[:, 512:] - codec.bf16_bits_to_f64(rope)) <= np.abs(codec.bf16_bits_to_f64(rope)) * 2.0 ** -8 + 1e-30)


def test_per_token_decode_matches_torch_sdpa():
    case, _, lat, rope = _small_case_cache(B=2, Q=2, H=4, topk=128, L=(500, 900), seed=13)
    cache = np.zeros((case.num_pages, 64, 672), np.uint8)
    fp8rows.write_cache_token(cache, lat, rope, np.arange(case.num_pages * 64))
    out, lse = fp8rows.sparse_decode_token(case.q_bits, cache, case.page_table, case.topk_indices,
                                           case.seq_lens, case.softmax_scale)
    q = codec.bf16_bits_to_f64(case.q_bits)
    for b in range(case.B):
        for j in range(case.Q):
            idx = case.topk_indices[b, j].astype(np.int64)
            rr = cache[case.page_table[b][idx // 64], idx % 64]
            s = torch.from_numpy(rr[:, 640:644].copy().view("<f4").astype(np.float64))
            lat_v = torch.from_numpy(rr[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64) * s
            rope_v = torch.from_numpy(rr[:, 512:640].copy()).view(torch.bfloat16).to(torch.float64) * s
            c = torch.cat([lat_v, rope_v], dim=1)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[b, j])[None, :, None, :], c[None, None].expand(1, case.H, -1, -1),
                c[None, None, :, :512].expand(1, case.H, -1, -1), scale=case.softmax_scale)
            np.testing.assert_allclose(out[b, j], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)
