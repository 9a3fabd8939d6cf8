"""Pins for the oracle's codecs and row encoding (CPU only).

Each test checks the oracle against something that is not the oracle: the
pages' printed row arithmetic, torch's float8_e4m3fn conversion (a library
round-to-nearest-even), exact rational brute force with fractions.Fraction,
and closed-form facts of the e2m1 grid.
"""
import bisect
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import codec, pack

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _finite_bf16_bits():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (b >> 7) & 0xFF
    return b[exp != 0xFF]


def _frac_of_bf16(bits):
    return Fraction(float(codec.bf16_bits_to_f64(np.array([bits], dtype=np.uint16))[0]))


def _e4m3_values_exact():
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


E4M3_EXACT = _e4m3_values_exact()
E2M1_EXACT = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def _rne_exact(mag: Fraction, grid):
    """Brute-force nearest-even rounding with exact rationals, saturating."""
    if mag >= grid[-1]:
        return len(grid) - 1
    i = bisect.bisect_left(grid, mag)
    if i < len(grid) and grid[i] == mag:
        return i
    lo, hi = i - 1, i
    dlo, dhi = mag - grid[lo], grid[hi] - mag
    if dlo < dhi:
        return lo
    if dhi < dlo:
        return hi
    return lo if lo % 2 == 0 else hi


def test_row_byte_arithmetic_matches_pages():
    g = {}
    with open(os.path.join(GOLDEN, "row_bytes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                g[k] = float(v)
    assert pack.D_LATENT == g["latent_values"] and pack.D_ROPE == g["rope_values"]
    assert pack.NIBBLE_BYTES == g["nvfp4_latent_bytes"] == pack.D_LATENT * 4 // 8
    assert pack.N_BLOCKS == g["nvfp4_scale_bytes"] == pack.D_LATENT // 16
    assert pack.ROW_BYTES - pack.ROPE_OFFSET == g["nvfp4_rope_bytes"]
    assert pack.ROW_BYTES == g["nvfp4_row_bytes"]
    assert pack.FP8_ROW_BYTES == g["fp8_row_bytes"] == g["fp8_latent_bytes"] + g["fp8_rope_bytes"]
    assert pack.ROW_BYTES + 2 * pack.FP8_ROW_BYTES == g["staged_bytes_per_row"]
    assert 100.0 * (pack.NIBBLE_BYTES + pack.N_BLOCKS) / g["fp8_latent_bytes"] == g["latent_ratio_percent"]
    rows = pack.encode_rows(np.zeros((3, 512), np.uint16), np.zeros((3, 64), np.uint16))
    assert rows.shape == (3, 352) and rows.dtype == np.uint8
    # every region starts on a 16-byte boundary and the row is 22 x 16 B
    assert pack.SCALE_OFFSET % 16 == 0 and pack.ROPE_OFFSET % 16 == 0 and pack.ROW_BYTES % 16 == 0


def test_e4m3_decode_matches_torch_all_bytes():
    codes = np.arange(256, dtype=np.uint8)
    ours = codec.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[m], ref[m])
    assert codec.E4M3_GRID[-1] == 448.0


def test_e4m3_encode_matches_torch_on_every_bf16():
    bits = _finite_bf16_bits()
    x = codec.bf16_bits_to_f64(bits)
    ours = codec.e4m3_encode(x)
    in_range = np.abs(x) < 464.0      # torch turns >= 464 into NaN; we saturate
    ref = torch.from_numpy(x[in_range].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours[in_range], ref)
    big = ~in_range
    np.testing.assert_array_equal(ours[big] & 0x7F, np.full(big.sum(), 0x7E, np.uint8))
    np.testing.assert_array_equal(ours[big] >> 7, np.signbit(x[big]).astype(np.uint8))


def test_block_scale_exhaustive_against_exact_rationals():
    """Every positive finite bf16 amax: scale byte == RNE_sat(amax/6) computed exactly."""
    bits = _finite_bf16_bits()
    bits = bits[bits < 0x8000]            # non-negative
    amax = codec.bf16_bits_to_f64(bits)
    blocks = np.zeros((bits.size, 16))
    blocks[:, 0] = amax
    rows = np.zeros((-(-bits.size // 32) * 32, 16))
    rows[:bits.size] = blocks
    ours = pack.block_scale_codes(rows.reshape(-1, 512)).reshape(-1)[:bits.size]
    for a, got in zip(amax.tolist(), ours.tolist()):
        want = _rne_exact(Fraction(a) / 6, E4M3_EXACT)
        assert got == want, (a, got, want)


def test_e2m1_against_exact_rationals_on_all_quotients_of_a_scale_sweep():
    """x/s for all bf16 x in the block's range and a spread of scales: codes equal
    exact-rational nearest-even rounding."""
    rng = np.random.default_rng(3)
    bits = _finite_bf16_bits()
    x_all = codec.bf16_bits_to_f64(bits)
    for s_code in [1, 7, 8, 0x1B, 0x30, 0x38, 0x3B, 0x3D, 0x4F, 0x55, 0x67, 0x7E]:
        s = float(codec.e4m3_decode(np.array([s_code]))[0])
        x = x_all[np.abs(x_all) <= 6 * s * 1.07]          # include a little saturation
        x = x if x.size <= 6000 else rng.choice(x, 6000, replace=False)
        with np.errstate(divide="ignore"):
            got = codec.e2m1_encode(x / s)
        for xi, g in zip(x.tolist(), got.tolist()):
            v = Fraction(xi) / Fraction(s)
            want = _rne_exact(abs(v), E2M1_EXACT) | (8 if np.signbit(xi) else 0)
            assert g == want, (xi, s, g, want)


def test_e2m1_tie_table_and_saturation():
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    want = [0, 2, 2, 4, 4, 6, 6]                     # codes: even code wins each tie
    assert codec.e2m1_encode(np.array(ties)).tolist() == want
    assert codec.e2m1_encode(-np.array(ties)).tolist() == [w | 8 for w in want]
    eps = 1e-9
    assert codec.e2m1_encode(np.array(ties) + eps).tolist() == [1, 2, 3, 4, 5, 6, 7]
    assert codec.e2m1_encode(np.array(ties) - eps).tolist() == [0, 1, 2, 3, 4, 5, 6]
    assert codec.e2m1_encode(np.array([6.0, 6.5, 1e9])).tolist() == [7, 7, 7]
    assert codec.e2m1_encode(np.array([-0.0, 0.0, -0.1])).tolist() == [8, 0, 8]


def test_grid_values_round_trip_exactly_for_every_scale():
    """Each e2m1 grid value times each positive finite E4M3 scale encodes back to
    itself, with the block scale recovered from amax = 6 * s."""
    scales = codec.e4m3_decode(np.arange(1, 0x7F))
    grid = np.concatenate([codec.E2M1_GRID, -codec.E2M1_GRID[1:]])     # 15 values
    lat = np.zeros((scales.size, 512))
    for i, s in enumerate(scales):
        blk = np.zeros(16)
        blk[0] = 6 * s
        blk[1:] = grid * s
        lat[i, :16] = blk
    sc = pack.block_scale_codes(lat)
    np.testing.assert_array_equal(sc[:, 0], np.arange(1, 0x7F))
    codes = pack.quantise_block_codes(lat, sc)
    want = codec.e2m1_encode(grid)
    for i in range(scales.size):
        np.testing.assert_array_equal(codes[i, 1:16], want)
        back = codec.e2m1_decode(codes[i, :16]) * scales[i]
        np.testing.assert_array_equal(back[1:], grid * scales[i])


def _bits(vals):
    from workloads import f32_to_bf16_bits
    return f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def test_special_blocks():
    from oracle.attention import dequant_rows
    lat = np.zeros((1, 512), np.float32)
    lat[0, 16:32] = -0.0                                # a negative-zero block
    lat[0, 32:48] = 3.0                                 # all equal
    lat[0, 48:64] = 0.01
    lat[0, 50] = 0.2                                    # one outlier x20
    lat[0, 64:80] = 1e-30                               # amax/6 far below the smallest subnormal scale
    lat[0, 80:96] = -1e-30
    rows = pack.encode_rows(_bits(lat), np.zeros((1, 64), np.uint16))
    scales = rows[0, 256:288]
    nib = rows[0, :256]
    codes = np.stack([nib & 0xF, nib >> 4], axis=1).reshape(-1)
    assert scales[0] == 0 and (codes[0:16] == 0).all()
    assert scales[1] == 0 and (codes[16:32] == 8).all()
    assert codec.e4m3_decode(scales[2:3])[0] == 0.5 and (codes[32:48] == 7).all()   # 3/6 = 0.5 exact
    s3 = codec.e4m3_decode(scales[3:4])[0]
    a = codec.bf16_bits_to_f64(_bits([0.2]))[0]
    assert Fraction(s3) == E4M3_EXACT[_rne_exact(Fraction(a) / 6, E4M3_EXACT)]
    assert codes[50] == _rne_exact(Fraction(a) / Fraction(s3), E2M1_EXACT)
    assert scales[4] == 0 and (codes[64:80] == 0).all() and (codes[80:96] == 8).all()
    deq = dequant_rows(rows)
    assert (deq[0, :16] == 0).all() and np.signbit(deq[0, 16:32]).all()
    assert (deq[0, 32:48] == 3.0).all()


def test_rope_bytes_are_e4m3_of_bf16_on_every_value():
    bits = _finite_bf16_bits()
    n = -(-bits.size // 64) * 64
    rope = np.zeros(n, np.uint16)
    rope[:bits.size] = bits
    rows = pack.encode_rows(np.zeros((n // 64, 512), np.uint16), rope.reshape(-1, 64))
    got = rows[:, 288:].reshape(-1)[:bits.size]
    x = codec.bf16_bits_to_f64(bits)
    m = np.abs(x) < 464
    ref = torch.from_numpy(x[m].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got[m], ref)


def test_nibble_order_low_then_high():
    lat = np.zeros((1, 512), np.float32)
    lat[0, 0] = 6.0   # amax of block 0 -> scale 1.0, code 7 at element 0
    lat[0, 1] = -1.0  # code 0xA at element 1
    rows = pack.encode_rows(_bits(lat), np.zeros((1, 64), np.uint16))
    assert rows[0, 0] == 0x7 | (0xA << 4)
    assert rows[0, 256] == 0x38            # E4M3 of 1.0


def test_write_cache_slots():
    cache = np.full((3, 64, 352), 0xCD, np.uint8)
    lat = _bits(np.ones((4, 512), np.float32))
    rope = _bits(np.ones((4, 64), np.float32))
    res = pack.write_cache(cache, lat, rope, [5, -1, 64 * 3, 130])
    assert res["bad_slots"] == 1
    assert (cache[0, 5] != 0xCD).any() and (cache[2, 2] != 0xCD).any()
    touched = np.zeros((3, 64), bool)
    touched[0, 5] = touched[2, 2] = True
    assert (cache[~touched] == 0xCD).all()


def test_bf16_bits_to_f64_matches_torch_on_every_pattern():
    """The bf16 decode every other pin builds on, against torch's own bfloat16 on all
    65,536 bit patterns (NaN patterns compare as NaN)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = codec.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_non_finite_inputs_follow_the_stated_reading():
    """NaN and infinity: a NaN latent value is left out of the block maximum and codes to
    magnitude 0 with its sign; an infinity saturates the scale to 448 and codes to +-6; rope
    NaN is E4M3 NaN with its sign, rope infinity +-448. Expected bytes written out by hand."""
    lat = np.zeros((1, 512), np.uint16)
    rope = np.zeros((1, 64), np.uint16)
    lat[0, 0:2] = [0x7FC0, 0x3F80]      # block 0: NaN, 1.0      -> scale E4M3(1/6) = 0x23 (0.171875)
    lat[0, 16:18] = [0x7F80, 0x3F80]    # block 1: +inf, 1.0     -> scale 448 (0x7E)
    lat[0, 32:34] = [0xFF80, 0x3F80]    # block 2: -inf, 1.0     -> scale 448
    lat[0, 48] = 0xFFC0                 # block 3: -NaN alone    -> amax 0, scale 0
    lat[0, 64:66] = [0x7FC1, 0xFFC0]    # block 4: NaNs only     -> scale 0
    rope[0, 0:4] = [0x7FC0, 0x7F80, 0xFF80, 0xFFC0]
    with np.errstate(all="ignore"):
        row = pack.encode_rows(lat, rope)[0]
    assert list(row[256:261]) == [0x23, 0x7E, 0x7E, 0x00, 0x00]
    # element codes (low nibble = even element): 1.0 / 0.171875 = 5.82 -> code 7 (6); NaN -> 0;
    # +inf -> 7 and 1/448 -> 0; -inf -> 0xF; -NaN -> 0x8; NaN -> 0 and -NaN -> 0x8
    assert row[0] == 0x70 and row[8] == 0x07 and row[16] == 0x0F and row[24] == 0x08 and row[32] == 0x80
    assert list(row[288:292]) == [0x7F, 0x7E, 0xFE, 0xFF]
    # the NaN-free elements of a block are coded as if the NaN were absent
    clean = lat.copy()
    clean[0, 0] = 0
    with np.errstate(all="ignore"):
        assert pack.encode_rows(clean, np.zeros((1, 64), np.uint16))[0][256] == 0x23
