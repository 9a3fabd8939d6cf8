"""Top-k position selection over indexer logits (oracle; test infrastructure only).

What the pages fix: decode attends only to the positions the indexer selected, up to 2,048 per
query token ("Prime Inference: serving GLM-5.3 to agents is a KV-cache problem", section
"Decode: TP4, and the copies it keeps": the top-2,048 positions; "Prime Inference", translated
page, "Native NVFP4 sparse MLA decode kernel": unused list entries are -1). The pages do not
define the indexer's logit formula, so the logits are an input here.

Readings (listed in the design notes):
  * query j of request b may select positions 0 .. seq_len[b] - Q + j (its causal range, the
    same rule the decode applies);
  * the K largest logits are selected; logits compare as floats, with NaN below every number
    and -0.0 below +0.0 (the order of their IEEE bit patterns read as sign-magnitude);
  * among equal logits the smaller position is taken first;
  * the selected positions are listed in increasing order; when fewer than K positions are in
    range, all of them are listed and the rest of the list is -1.
"""
from __future__ import annotations

import numpy as np


def order_keys(logits: np.ndarray) -> np.ndarray:
    """uint32 keys whose unsigned order is the selection order of float32 logits: for x < y
    (as floats, -0.0 < +0.0) key(x) < key(y); every NaN gets key 0, below all numbers."""
    x = np.ascontiguousarray(logits, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    neg = (b >> 31) == 1
    k = np.where(neg, (~b) & 0xFFFFFFFF, b | 0x80000000)
    k = np.where(np.isnan(x), 0, k)
    return k.astype(np.uint32)


def select_row(logits_row: np.ndarray, n_valid: int, K: int) -> np.ndarray:
    """The K selected positions of one query (int32 [K], increasing, -1 padded)."""
    n = max(0, min(int(n_valid), logits_row.shape[0]))
    out = np.full(K, -1, dtype=np.int32)
    if n == 0:
        return out
    keys = order_keys(logits_row[:n]).astype(np.int64)
    pos = np.arange(n, dtype=np.int64)
    # rank by (key descending, position ascending) and keep the first K
    order = np.lexsort((pos, -keys))
    take = np.sort(order[:K])
    out[:take.size] = take
    return out


def select(logits: np.ndarray, seq_lens: np.ndarray, Q: int, K: int) -> np.ndarray:
    """logits float32 [B, Q, S] (S >= the longest range), seq_lens int [B] -> int32 [B, Q, K]."""
    B = logits.shape[0]
    out = np.empty((B, Q, K), dtype=np.int32)
    for b in range(B):
        for j in range(Q):
            out[b, j] = select_row(logits[b, j], int(seq_lens[b]) - Q + j + 1, K)
    return out
