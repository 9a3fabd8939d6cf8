"""NVFP4 row encoding and the paged cache write (oracle; test infrastructure only).

What a row holds, from "Prime Inference" (translated page), section "Making
room for low-latency decode": the 512-value MLA latent in NVFP4 (four bits per
value, one FP8 scale per group of 16 values) and the 64-value rope part in
FP8, 352 bytes per row instead of 576. The byte split 256 + 32 + 64 is the
table in "Prime Inference: serving GLM-5.3 to agents is a KV-cache problem",
section "Four bits per latent value: where 352 comes from"; that table also
implies there is no per-row or per-tensor scale (the row has no bytes left for
one), so the rope bytes are plain E4M3 of the bf16 values.

Readings where the pages are silent (each is listed in the design notes):
  * block scale s = E4M3(amax / 6) with amax the largest |value| of the block,
    6 being the largest e2m1 magnitude; amax/6 is rounded once, from its exact
    value, to nearest-even and saturated at 448;
  * element code = e2m1(x / s) using the rounded scale, nearest-even,
    saturating at 6, sign kept; if s == 0 every magnitude code is 0;
  * byte layout: bytes [0,256) hold element 2i in the low nibble and 2i+1 in
    the high nibble of byte i; bytes [256,288) hold the 32 block scales in
    order; bytes [288,352) hold the 64 rope bytes;
  * non-finite inputs: a NaN latent value takes no part in its block's
    maximum and is coded with magnitude 0 (its sign bit kept); an infinity
    takes part, so its block scale saturates to 448 and it codes as +-6; a
    rope NaN becomes E4M3 NaN (0x7F, sign kept) and a rope infinity +-448;
  * the cache is uint8 [num_pages, 64, 352]; a slot s addresses page s // 64,
    row s % 64; slot -1 means "skip this token"; any other slot outside
    [0, num_pages*64) is also skipped (and counted as a bad slot).
"""
from __future__ import annotations

import numpy as np

from . import codec

D_LATENT = 512
D_ROPE = 64
BLOCK = 16
N_BLOCKS = D_LATENT // BLOCK          # 32 scales
NIBBLE_BYTES = D_LATENT // 2          # 256
SCALE_OFFSET = NIBBLE_BYTES           # 256
ROPE_OFFSET = SCALE_OFFSET + N_BLOCKS  # 288
ROW_BYTES = ROPE_OFFSET + D_ROPE      # 352
FP8_ROW_BYTES = D_LATENT + D_ROPE     # 576
PAGE_TOKENS = 64


def block_scale_codes(latent: np.ndarray) -> np.ndarray:
    """E4M3 scale byte of each 16-value block: E4M3_rn_sat(amax / 6).

    latent: float64 [N, 512] (exact bf16 values). Returns uint8 [N, 32].

    amax / 6 is formed in float64. Its exact value is either a float64 number
    (amax divisible by 3 in the binary sense) or has a repeating binary
    expansion (...0101...), which is never within float64 rounding distance of
    an E4M3 midpoint; so rounding the float64 quotient gives the same E4M3 code
    as rounding the exact quotient.
    """
    x = np.asarray(latent, dtype=np.float64).reshape(-1, N_BLOCKS, BLOCK)
    # Reading for non-finite values: a NaN takes no part in its block's maximum
    # (a block of NaNs and zeros has amax 0); an infinity does, and amax/6 =
    # inf then saturates the scale to 448.
    amax = np.where(np.isnan(x), 0.0, np.abs(x)).max(axis=2)
    return codec.e4m3_encode(amax / 6.0)


def quantise_block_codes(latent: np.ndarray, scale_codes: np.ndarray) -> np.ndarray:
    """e2m1 codes of every latent value given its block's scale byte.

    latent float64 [N, 512], scale_codes uint8 [N, 32] -> uint8 [N, 512] codes.
    v = x / s with s the decoded (rounded) scale. As for the scale, the exact
    quotient of a bf16 value by an E4M3 value is either exact in float64 or
    far from every e2m1 midpoint, so the float64 quotient rounds the same way.
    """
    x = np.asarray(latent, dtype=np.float64).reshape(-1, N_BLOCKS, BLOCK)
    s = codec.e4m3_decode(scale_codes).reshape(-1, N_BLOCKS, 1)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = np.where(s > 0, x / np.where(s > 0, s, 1.0), 0.0 * x)   # 0*x keeps the sign of x
    codes = codec.e2m1_encode(v)
    return codes.reshape(-1, D_LATENT)


def encode_rows(latent_bits: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """Encode bf16 rows into 352-byte NVFP4 rows.

    latent_bits uint16 [N, 512], rope_bits uint16 [N, 64] (bf16 bit patterns)
    -> uint8 [N, 352].
    """
    lat = codec.bf16_bits_to_f64(latent_bits).reshape(-1, D_LATENT)
    rope = codec.bf16_bits_to_f64(rope_bits).reshape(-1, D_ROPE)
    n = lat.shape[0]
    scales = block_scale_codes(lat)
    codes = quantise_block_codes(lat, scales).astype(np.uint8)
    row = np.zeros((n, ROW_BYTES), dtype=np.uint8)
    row[:, :NIBBLE_BYTES] = codes[:, 0::2] | (codes[:, 1::2] << 4)
    row[:, SCALE_OFFSET:ROPE_OFFSET] = scales
    row[:, ROPE_OFFSET:] = codec.e4m3_encode(rope)
    return row


def write_cache(cache: np.ndarray, latent_bits, rope_bits, slot_mapping) -> dict:
    """Write encoded rows into a paged cache in place, following slot_mapping.

    cache: uint8 [num_pages, 64, 352]. Returns {"bad_slots": count} for slots
    other than -1 that fall outside the cache (those rows are not written).
    When two tokens map to the same slot, the later one in token order is what
    this oracle leaves; callers that compare against a parallel writer should
    not map two tokens to one slot.
    """
    num_pages = cache.shape[0]
    rows = encode_rows(latent_bits, rope_bits)
    slots = np.asarray(slot_mapping, dtype=np.int64).reshape(-1)
    bad = 0
    for t, s in enumerate(slots):
        if s == -1:
            continue
        if s < 0 or s >= num_pages * PAGE_TOKENS:
            bad += 1
            continue
        cache[s // PAGE_TOKENS, s % PAGE_TOKENS] = rows[t]
    return {"bad_slots": bad}
