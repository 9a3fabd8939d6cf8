"""FP8 576-byte rows and the staged NVFP4 -> FP8 copy (oracle; test infrastructure only).

What the pages fix:
  * an FP8 cache row holds 576 bytes: one byte per value of the 512-value latent and the 64-value
    rope key ("Prime Inference: serving GLM-5.3 to agents is a KV-cache problem", section "Four
    bits per latent value: where 352 comes from", the FP8-row column of its table; the translated
    "Prime Inference" page, "Making room for low-latency decode": 576 -> 352 bytes);
  * the staged path reads each selected 352-byte NVFP4 row, writes a 576-byte FP8 copy to GPU
    memory, and an FP8 attention kernel reads that copy: 352 + 576 + 576 = 1,504 bytes per
    selected row, against 352 for the native kernel (same page, section "A kernel that reads
    four bits directly", and the translated page, "Native NVFP4 sparse MLA decode kernel");
  * every path computes the same attention (oracle.attention), only over differently rounded
    rows.

  * TokenSpeed's per-token FP8 cache (the "TokenSpeed" walkthrough, section 8 "MLA KV layout", its
    per_token_head write path): the latent is stored as FP8 E4M3 of latent / scale with one fp32
    scale = max(amax, 1e-26) / 448 per token (amax the largest |latent value|), computed in fp32;
    the rope part is divided by the same scale and kept in the model dtype (bf16).

Readings (listed in the design notes):
  * an FP8 row is E4M3 of each value (codec.e4m3_encode: nearest, ties to even, saturating at
    +-448, NaN kept as 0x7F with its sign), latent in bytes 0..511, rope in bytes 512..575, and no
    scale (the 576 bytes leave none);
  * the staged copy of an NVFP4 row rounds each dequantised latent value e2m1(code) * E4M3(scale)
    (exact in float64) once to E4M3 the same way, so values past 448 saturate; the rope bytes are
    E4M3 already and are copied unchanged; a block whose scale byte is the E4M3 NaN (0x7F or 0xFF,
    which pack never writes) stages as 0x7F for each of its 16 values;
  * the staging of one decode step writes, for query (b, j) and list entry i, the copy of the
    selected row to staged row (b*Q + j)*K + i and makes the FP8 decode's list entry i equal to i
    when the entry is usable under the decode's rule (oracle.attention.valid_entries), else -1;
    staged rows of unusable entries are not written. The FP8 decode then runs over the staged
    rows as B*Q one-query requests of length K whose page table is the identity;
  * the per-token FP8 row (GB300 layout of TokenSpeed's three buffers) is 672 bytes: bytes
    0..511 the E4M3 latent codes, 512..639 the 64 bf16 rope values, 640..643 the fp32 scale
    (little-endian), 644..671 zero; one row keeps a token's bytes together for one gather, and
    four rows are a whole number of 128-byte units. The arithmetic follows TokenSpeed's write
    path: amax, the scale and both divisions in fp32 (IEEE, round to nearest even), then E4M3
    (nearest even, saturating) and bf16 (nearest even) rounding. Dequantised values are
    E4M3(code) * scale and bf16(rope) * scale (exact in float64).
"""
from __future__ import annotations

import numpy as np

from . import codec
from .attention import D_QK, attend, dequant_rows, valid_entries
from .pack import (BLOCK, D_LATENT, D_ROPE, FP8_ROW_BYTES, N_BLOCKS, PAGE_TOKENS, ROPE_OFFSET, ROW_BYTES,
                   SCALE_OFFSET)


def encode_rows_fp8(latent_bits: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16 [N, 512], [N, 64]) -> FP8 rows uint8 [N, 576]."""
    lat = codec.bf16_bits_to_f64(np.asarray(latent_bits, dtype=np.uint16).reshape(-1, D_LATENT))
    rope = codec.bf16_bits_to_f64(np.asarray(rope_bits, dtype=np.uint16).reshape(-1, D_ROPE))
    return np.concatenate([codec.e4m3_encode(lat), codec.e4m3_encode(rope)], axis=1)


def dequant_rows_fp8(rows: np.ndarray) -> np.ndarray:
    """FP8 rows uint8 [..., 576] -> float64 [N, 576]."""
    rows = np.asarray(rows, dtype=np.uint8).reshape(-1, FP8_ROW_BYTES)
    return codec.e4m3_decode(rows)


def stage_rows(rows: np.ndarray) -> np.ndarray:
    """352-byte NVFP4 rows -> their 576-byte FP8 copies (latent re-rounded, rope bytes copied)."""
    rows = np.asarray(rows, dtype=np.uint8).reshape(-1, ROW_BYTES)
    lat = codec.e4m3_encode(dequant_rows(rows)[:, :D_LATENT])
    nan_scale = (rows[:, SCALE_OFFSET:SCALE_OFFSET + N_BLOCKS] & 0x7F) == 0x7F
    lat = np.where(np.repeat(nan_scale, BLOCK, axis=1), np.uint8(0x7F), lat)
    return np.concatenate([lat, rows[:, ROPE_OFFSET:ROPE_OFFSET + D_ROPE]], axis=1)


def write_cache_fp8(cache: np.ndarray, latent_bits, rope_bits, slot_mapping) -> None:
    """Write FP8 rows into cache uint8 [num_pages, 64, 576] at the slots (slot -1, or any slot
    outside the cache, is skipped)."""
    rows = encode_rows_fp8(latent_bits, rope_bits)
    flat = cache.reshape(-1, FP8_ROW_BYTES)
    for r, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if 0 <= s < flat.shape[0]:
            flat[s] = rows[r]


def stage(cache, page_table, topk_indices, seq_lens, Q: int):
    """The staging of one decode step over an NVFP4 cache.

    Returns (staged uint8 [B*Q*K, 576] with unwritten rows zero, written bool [B*Q*K],
    fp8_topk int32 [B*Q, 1, K], fp8_page_table int32 [B*Q, K/64 rounded up], fp8_seq_lens int32
    [B*Q]): the inputs of the FP8 decode over the staged rows.
    """
    B = topk_indices.shape[0]
    K = topk_indices.shape[2]
    num_pages = cache.shape[0]
    staged = np.zeros((B * Q * K, FP8_ROW_BYTES), dtype=np.uint8)
    written = np.zeros(B * Q * K, dtype=bool)
    new_topk = np.full((B * Q, 1, K), -1, dtype=np.int32)
    for b in range(B):
        L = int(seq_lens[b])
        for j in range(Q):
            u = b * Q + j
            idx = np.asarray(topk_indices[b, j], dtype=np.int64)
            ok = valid_entries(idx, L, L - Q + j, page_table[b], num_pages)
            sel = np.nonzero(ok)[0]
            if sel.size:
                pages = np.asarray(page_table[b], dtype=np.int64)[idx[sel] // PAGE_TOKENS]
                staged[u * K + sel] = stage_rows(cache[pages, idx[sel] % PAGE_TOKENS])
                written[u * K + sel] = True
                new_topk[u, 0, sel] = sel
    pages_per_unit = -(-K // PAGE_TOKENS)
    # the identity page table: unit u's list entry i lives on staged page u*pages_per_unit + i//64
    # (staged rows are K apart per unit; K is a multiple of 64 in every staged call)
    pt = (np.arange(B * Q, dtype=np.int64)[:, None] * pages_per_unit
          + np.arange(pages_per_unit, dtype=np.int64)[None, :]).astype(np.int32)
    return staged, written, new_topk, pt, np.full(B * Q, K, dtype=np.int32)


TOKEN_ROW_BYTES = 672
TOKEN_ROPE_OFFSET = 512
TOKEN_SCALE_OFFSET = 640


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values -> bf16 bit patterns, round to nearest even (NaN kept as a quiet NaN)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    nan = np.isnan(x)
    return np.where(nan, (b >> 16) | 0x40, rounded).astype(np.uint16)


def encode_rows_token(latent_bits: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16 [N, 512], [N, 64]) -> per-token FP8 rows uint8 [N, 672]."""
    lat = codec.bf16_bits_to_f64(np.asarray(latent_bits, dtype=np.uint16).reshape(-1, D_LATENT)).astype(np.float32)
    rope = codec.bf16_bits_to_f64(np.asarray(rope_bits, dtype=np.uint16).reshape(-1, D_ROPE)).astype(np.float32)
    n = lat.shape[0]
    amax = np.abs(lat).max(axis=1, keepdims=True)                     # fp32, exact
    scale = (np.maximum(amax, np.float32(1e-26)) / np.float32(448.0)).astype(np.float32)
    codes = codec.e4m3_encode((lat / scale).astype(np.float32).astype(np.float64))
    rope_bf = _f32_to_bf16_bits((rope / scale).astype(np.float32))
    rows = np.zeros((n, TOKEN_ROW_BYTES), dtype=np.uint8)
    rows[:, :D_LATENT] = codes
    rows[:, TOKEN_ROPE_OFFSET:TOKEN_SCALE_OFFSET] = rope_bf.view(np.uint8).reshape(n, 2 * D_ROPE)
    rows[:, TOKEN_SCALE_OFFSET:TOKEN_SCALE_OFFSET + 4] = scale.astype('<f4').view(np.uint8).reshape(n, 4)
    return rows


def dequant_rows_token(rows: np.ndarray) -> np.ndarray:
    """Per-token FP8 rows uint8 [..., 672] -> float64 [N, 576]."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.uint8).reshape(-1, TOKEN_ROW_BYTES))
    scale = rows[:, TOKEN_SCALE_OFFSET:TOKEN_SCALE_OFFSET + 4].copy().view('<f4').astype(np.float64)   # [N, 1]
    lat = codec.e4m3_decode(rows[:, :D_LATENT]) * scale
    rope_bits = rows[:, TOKEN_ROPE_OFFSET:TOKEN_SCALE_OFFSET].copy().view('<u2')
    rope = codec.bf16_bits_to_f64(rope_bits) * scale
    return np.concatenate([lat, rope], axis=1)


def write_cache_token(cache: np.ndarray, latent_bits, rope_bits, slot_mapping) -> None:
    """Write per-token FP8 rows into cache uint8 [num_pages, 64, 672] at the slots (slot -1, or any
    slot outside the cache, is skipped)."""
    rows = encode_rows_token(latent_bits, rope_bits)
    flat = cache.reshape(-1, TOKEN_ROW_BYTES)
    for r, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if 0 <= s < flat.shape[0]:
            flat[s] = rows[r]


def sparse_decode_token(q_bits, cache, page_table, topk_indices, seq_lens, scale, units=None):
    """Sparse MLA decode over a paged per-token FP8 cache uint8 [num_pages, 64, 672]; the same
    rules and outputs as attention.sparse_decode."""
    return _sparse_decode_rows(q_bits, cache, page_table, topk_indices, seq_lens, scale, units,
                               dequant_rows_token, TOKEN_ROW_BYTES)


def sparse_decode_fp8(q_bits, cache, page_table, topk_indices, seq_lens, scale, units=None):
    """Sparse MLA decode over a paged FP8 cache uint8 [num_pages, 64, 576]; the same rules and
    outputs as attention.sparse_decode."""
    return _sparse_decode_rows(q_bits, cache, page_table, topk_indices, seq_lens, scale, units,
                               dequant_rows_fp8, FP8_ROW_BYTES)


def _sparse_decode_rows(q_bits, cache, page_table, topk_indices, seq_lens, scale, units, dequant, row_bytes):
    q = codec.bf16_bits_to_f64(q_bits)
    B, Q, H, _ = q.shape
    num_pages = cache.shape[0]
    out = np.full((B, Q, H, D_LATENT), np.nan)
    lse = np.full((B, Q, H), np.nan)
    todo = [(b, j) for b in range(B) for j in range(Q)] if units is None else list(units)
    for b, j in todo:
        L = int(seq_lens[b])
        idx = np.asarray(topk_indices[b, j], dtype=np.int64)
        ok = valid_entries(idx, L, L - Q + j, page_table[b], num_pages)
        sel = idx[ok]
        pages = np.asarray(page_table[b], dtype=np.int64)[sel // PAGE_TOKENS]
        c = dequant(cache[pages, sel % PAGE_TOKENS]) if sel.size else np.zeros((0, D_QK))
        out[b, j], lse[b, j] = attend(q[b, j], c, scale)
    return out, lse
