"""Dequantisation and sparse / dense MLA decode in fp64 (oracle; test infrastructure only).

What is computed, from the pages:
  * one cache row per token holds a 512-value latent and a 64-value rope key;
    every head reads the same row ("Prime Inference: serving GLM-5.3 to agents
    is a KV-cache problem", section "Prefill topology: why DEP8 holds five
    times the cache");
  * the decode kernel loads the rows the indexer selected, unpacks them and
    computes attention with FP16 operands and FP32 accumulation; the staged,
    native and FP8 kernels all compute the same attention ("Prime Inference",
    translated page, subsection "Native NVFP4 sparse MLA decode kernel"); so
    the oracle is plain softmax attention over the dequantised rows;
  * each query reads at most 2,048 selected positions; unused list entries are
    -1 and must not be read (same subsection; and "Decode: TP4, and the
    copies it keeps" on the second page);
  * softmax scale 1/sqrt(192) = 0.07216882 (TokenSpeed walkthrough, MLA
    decode benchmark example).

Readings (listed in the design notes):
  * q is the absorbed query: its first 512 values meet the latent, its last 64
    the rope key; the value vector is the dequantised latent itself;
  * an index entry is used only if 0 <= idx < seq_len[b], idx is at or before
    the query's causal position seq_len[b] - Q + j, idx // 64 is a column of
    the page table and that page-table entry is in [0, num_pages); every other
    entry (including -1) is left out of the softmax entirely;
  * duplicate entries count as many times as they are listed;
  * LSE is the natural log of the softmax denominator, scale included; a
    query with no usable entry gets out = 0 and LSE = -inf.
"""
from __future__ import annotations

import numpy as np

from . import codec
from .pack import D_LATENT, D_ROPE, N_BLOCKS, BLOCK, NIBBLE_BYTES, SCALE_OFFSET, ROPE_OFFSET, PAGE_TOKENS

D_QK = D_LATENT + D_ROPE


def dequant_rows(rows: np.ndarray) -> np.ndarray:
    """352-byte rows -> float64 [N, 576]: e2m1(code) * E4M3(scale) for the
    latent, E4M3(byte) for the rope part."""
    rows = np.asarray(rows, dtype=np.uint8).reshape(-1, rows.shape[-1])
    nib = rows[:, :NIBBLE_BYTES].astype(np.int64)
    codes = np.empty((rows.shape[0], D_LATENT), dtype=np.int64)
    codes[:, 0::2] = nib & 0xF
    codes[:, 1::2] = nib >> 4
    scale = codec.e4m3_decode(rows[:, SCALE_OFFSET:SCALE_OFFSET + N_BLOCKS])
    lat = codec.e2m1_decode(codes) * np.repeat(scale, BLOCK, axis=1)
    rope = codec.e4m3_decode(rows[:, ROPE_OFFSET:ROPE_OFFSET + D_ROPE])
    return np.concatenate([lat, rope], axis=1)


def valid_entries(idx, seq_len: int, causal_pos: int, page_row, num_pages: int) -> np.ndarray:
    """Mask of usable index entries for one query (see module docstring)."""
    idx = np.asarray(idx, dtype=np.int64)
    ok = (idx >= 0) & (idx < seq_len) & (idx <= causal_pos)
    col = np.where(ok, idx // PAGE_TOKENS, 0)
    ok &= col < len(page_row)
    pg = np.asarray(page_row, dtype=np.int64)[np.clip(col, 0, len(page_row) - 1)]
    ok &= (pg >= 0) & (pg < num_pages)
    return ok


def attend(q: np.ndarray, c: np.ndarray, scale: float):
    """Softmax attention of q [H, 576] over dequantised rows c [n, 576].

    Returns (out float64 [H, 512], lse float64 [H]). n == 0 gives zeros / -inf.
    """
    H = q.shape[0]
    if c.shape[0] == 0:
        return np.zeros((H, D_LATENT)), np.full(H, -np.inf)
    z = scale * (q @ c.T)                      # [H, n]
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ c[:, :D_LATENT]) / l
    return out, (m + np.log(l))[:, 0]


def sparse_decode(q_bits, cache, page_table, topk_indices, seq_lens, scale, units=None):
    """Sparse MLA decode over the paged NVFP4 cache.

    q_bits uint16 [B, Q, H, 576] (bf16), cache uint8 [num_pages, 64, 352],
    page_table int [B, max_pages], topk_indices int [B, Q, K], seq_lens int [B].
    units: optional iterable of (b, j) to compute; others are left as NaN.
    Returns (out float64 [B, Q, H, 512], lse float64 [B, Q, H]).
    """
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
        rows = cache[pages, sel % PAGE_TOKENS]
        c = dequant_rows(rows) if sel.size else np.zeros((0, D_QK))
        out[b, j], lse[b, j] = attend(q[b, j], c, scale)
    return out, lse


def dense_decode(q_bits, cache, page_table, seq_lens, scale):
    """Dense control: every query attends to all positions 0..seq_len-1 of its
    request (no index list, no causal offset within the step)."""
    q = codec.bf16_bits_to_f64(q_bits)
    B, Q, H, _ = q.shape
    out = np.zeros((B, Q, H, D_LATENT))
    lse = np.zeros((B, Q, H))
    for b in range(B):
        L = int(seq_lens[b])
        pos = np.arange(L)
        pages = np.asarray(page_table[b], dtype=np.int64)[pos // PAGE_TOKENS]
        c = dequant_rows(cache[pages, pos % PAGE_TOKENS])
        for j in range(Q):
            out[b, j], lse[b, j] = attend(q[b, j], c, scale)
    return out, lse
