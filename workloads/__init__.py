"""Seeded synthetic inputs for the NVFP4 sparse MLA decode path.

This module only draws random numbers and lays out index structures. It holds
none of the method's arithmetic (no quantisation, no attention), so both the
CPU oracle and the CUDA path can take their inputs from it.

Shapes follow the workloads on the "Prime Inference" pages (decode section,
"Making room for low-latency decode" and "Native NVFP4 sparse MLA decode
kernel"): a 512-value MLA latent plus a 64-value RoPE key per cached token,
64-token pages, and up to 2,048 indexer-selected positions per query token.
The five cases are:

  0 tiny            B=1,  Q=1, H=16, L=4,096,  top-k 256
  1 decode shard    B=16, Q=1, H=32, L=140,000, top-k 2,048 (half from the last 4K)
  2 mixed agent     B=64, Q=1, H=32, L~U[70K,160K], top-k 2,048
  3 spec verify     B=32, Q=4, H=32, L_ctx~U[100K,150K] + 6,000 packed rows
  4 capacity        B=128, Q=1, H=32, 1.63M-token shared pool, lognormal L
  3s spec verify, shared lists: case 3 with the 4 draft tokens' index lists sharing 90 % of
                    their positions (one request-level set plus 10 % of each token's own)
  4d dense control  B=8, Q=1, H=32, L=8,000, top-k = every position in order

Row values: latent = N(0,1) * c_d with c_d ~ lognormal(0, 0.5) per channel,
each element multiplied by 20 with probability 0.001; rope ~ N(0,1);
q ~ N(0,1). Everything is rounded to bf16 (round to nearest even) and handled
as raw uint16 bit patterns on the host.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE_TOKENS = 64
D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)   # 128 nope + 64 rope dims
OUTLIER_PROB = 1e-3
OUTLIER_GAIN = 20.0

CONFIG_NAMES = {
    0: "tiny B=1 H=16 L=4096 topk=256",
    1: "decode-shard B=16 H=32 L=140000 topk=2048",
    2: "mixed-agent B=64 H=32 L~U[70K,160K] topk=2048",
    3: "spec-verify B=32 Q=4 H=32 L~U[100K,150K]+6000 topk=2048",
    4: "capacity B=128 H=32 pool=1.63M tokens topk=2048",
    "4d": "dense-control B=8 H=32 L=8000 topk=8000",
    "3s": "spec-verify-shared B=32 Q=4 H=32 L~U[100K,150K]+6000 topk=2048, lists 90% shared",
}
SHARED_FRACTION = 0.9   # case 3s: fraction of a draft token's list taken from the request's shared set


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


@dataclasses.dataclass
class DecodeCase:
    """Index structures and queries for one decode step, plus how to draw rows."""
    name: str
    B: int
    Q: int
    H: int
    topk: int
    num_pages: int
    seq_lens: np.ndarray          # int32 [B]
    page_table: np.ndarray        # int32 [B, max_pages]
    topk_indices: np.ndarray      # int32 [B, Q, topk], logical positions, -1 = unused
    q_bits: np.ndarray            # uint16 [B, Q, H, 576] (bf16 bit patterns)
    channel_scale: np.ndarray     # float32 [512], the per-channel c_d
    row_seed: int                 # seeds the cache-row contents per physical page
    softmax_scale: float = SOFTMAX_SCALE
    # spec-verify only: rows written by mla_kv_pack in the same step
    new_slots: Optional[np.ndarray] = None   # int64 [N_new]
    notes: dict = dataclasses.field(default_factory=dict)

    @property
    def units(self) -> int:
        return self.B * self.Q

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]


def _channel_scale(rng: np.random.Generator) -> np.ndarray:
    return rng.lognormal(0.0, 0.5, size=D_LATENT).astype(np.float32)


def _queries(rng: np.random.Generator, B: int, Q: int, H: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((B, Q, H, D_QK), dtype=np.float32))


def _draw_without_replacement(rng, lo: int, hi: int, n: int) -> np.ndarray:
    """n distinct integers uniform in [lo, hi)."""
    return (lo + rng.choice(hi - lo, size=n, replace=False)).astype(np.int64)


def _shared_lists(rng, L: int, Q: int, K: int, shared: float) -> np.ndarray:
    """Index lists [Q, K] of one request whose Q query tokens share most positions, as the draft
    tokens of a speculative-verify step do: a set of K positions valid for every token (before
    L - Q + 1); token j keeps round(shared * K) of them (its own random choice) and draws the rest
    from its own causal range outside the set. Each list is in increasing position order (the
    order a top-k selection writes)."""
    base = _draw_without_replacement(rng, 0, L - Q + 1, K)
    n_keep = int(round(shared * K))
    out = np.empty((Q, K), dtype=np.int64)
    for j in range(Q):
        hi = L - Q + j + 1
        keep = base[rng.permutation(K)[:n_keep]]
        rest = np.setdiff1d(np.arange(hi, dtype=np.int64), base, assume_unique=True)
        own = rest[rng.choice(rest.size, size=K - n_keep, replace=False)]
        out[j] = np.sort(np.concatenate([keep, own]))
    return out


def subset_lists(rng, L: int, Q: int, K: int, keep: float) -> np.ndarray:
    """Index lists [Q, K] of one request whose Q query tokens each keep round(keep * K) positions
    of one set of K positions valid for all of them (before L - Q + 1), in increasing order and -1
    padded: the tokens' lists fit in one shared list of K entries."""
    base = np.sort(_draw_without_replacement(rng, 0, L - Q + 1, K))
    n = int(round(keep * K))
    out = np.full((Q, K), -1, dtype=np.int64)
    for j in range(Q):
        out[j, :n] = np.sort(base[rng.permutation(K)[:n]])
    return out


def fold_lists(topk_indices: np.ndarray):
    """Per-query index lists int [B, Q, K] -> (shared int32 [B, U], member uint8 [B, U]): each
    request's distinct entries (-1 dropped; invalid positions kept, the decode skips them) in
    increasing order, -1 padded to the longest union U, and bit j of member set where the entry
    is in query j's list."""
    B, Q, _ = topk_indices.shape
    unions = [np.unique(topk_indices[b][topk_indices[b] != -1]) for b in range(B)]
    U = max(1, max(u.size for u in unions))
    shared = np.full((B, U), -1, dtype=np.int32)
    member = np.zeros((B, U), dtype=np.uint8)
    for b, u in enumerate(unions):
        shared[b, :u.size] = u
        for j in range(Q):
            member[b, :u.size] |= (np.isin(u, topk_indices[b, j]).astype(np.uint8) << j)
    return shared, member


def host_rows(case: DecodeCase, pages: np.ndarray):
    """Draw the bf16 latent and rope rows of the given physical pages on the host.

    Each page has its own generator (seeded by (row_seed, page)), so any page
    can be regenerated alone. Returns (latent_bits uint16 [n*64, 512],
    rope_bits uint16 [n*64, 64]) in page order.
    """
    pages = np.asarray(pages, dtype=np.int64).reshape(-1)
    lat = np.empty((pages.size * PAGE_TOKENS, D_LATENT), dtype=np.uint16)
    rope = np.empty((pages.size * PAGE_TOKENS, D_ROPE), dtype=np.uint16)
    for i, p in enumerate(pages):
        rng = np.random.default_rng([case.row_seed, int(p)])
        x = rng.standard_normal((PAGE_TOKENS, D_LATENT), dtype=np.float32) * case.channel_scale
        gain = np.where(rng.random((PAGE_TOKENS, D_LATENT)) < OUTLIER_PROB, OUTLIER_GAIN, 1.0)
        lat[i * PAGE_TOKENS:(i + 1) * PAGE_TOKENS] = f32_to_bf16_bits((x * gain).astype(np.float32))
        r = rng.standard_normal((PAGE_TOKENS, D_ROPE), dtype=np.float32)
        rope[i * PAGE_TOKENS:(i + 1) * PAGE_TOKENS] = f32_to_bf16_bits(r)
    return lat, rope


def device_rows(case: DecodeCase, n_rows: int, device, seed_offset: int = 0):
    """Draw n_rows bf16 latent/rope rows directly on a torch device.

    Same distributions as host_rows, drawn with torch's generator on the
    device (the values differ from host_rows; use one or the other within a
    test). Returns (latent bf16 [n_rows, 512], rope bf16 [n_rows, 64]).
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(case.row_seed) * 1000003 + seed_offset)
    c = torch.as_tensor(case.channel_scale, device=device)
    lat = torch.empty((n_rows, D_LATENT), dtype=torch.bfloat16, device=device)
    rope = torch.empty((n_rows, D_ROPE), dtype=torch.bfloat16, device=device)
    chunk = 1 << 18
    for s in range(0, n_rows, chunk):
        n = min(chunk, n_rows - s)
        x = torch.randn((n, D_LATENT), generator=g, device=device) * c
        u = torch.rand((n, D_LATENT), generator=g, device=device)
        x = torch.where(u < OUTLIER_PROB, x * OUTLIER_GAIN, x)
        lat[s:s + n] = x.to(torch.bfloat16)
        rope[s:s + n] = torch.randn((n, D_ROPE), generator=g, device=device).to(torch.bfloat16)
    return lat, rope


def _pages_for(lengths, perm, cycle=False):
    """Assign physical pages to each request from a permuted pool."""
    rows = []
    off = 0
    for L in lengths:
        n = -(-int(L) // PAGE_TOKENS)
        if cycle:
            idx = (off + np.arange(n)) % perm.size
        else:
            idx = off + np.arange(n)
        rows.append(perm[idx])
        off += n
    width = max(r.size for r in rows)
    table = np.full((len(rows), width), -1, dtype=np.int32)
    for b, r in enumerate(rows):
        table[b, :r.size] = r
    return table, off


def make_case(cfg, seed: Optional[int] = None) -> DecodeCase:
    """Build the index structures and queries of one case (cfg in 0..4 or '4d')."""
    if seed is None:
        seed = {"4d": 1504, "3s": 1703}.get(cfg, 1000 + (int(cfg) if cfg not in ("4d", "3s") else 0))
    rng = np.random.default_rng(seed)
    c = _channel_scale(rng)
    row_seed = int(rng.integers(1, 2**31 - 1))

    if cfg == 0:
        B, Q, H, K = 1, 1, 16, 256
        L = np.array([4096], dtype=np.int64)
        num_pages = 64
        perm = rng.permutation(num_pages).astype(np.int32)
        table, _ = _pages_for(L, perm)
        topk = _draw_without_replacement(rng, 0, 4096, K).reshape(1, 1, K)
        notes = {}
    elif cfg == 1:
        B, Q, H, K = 16, 1, 32, 2048
        L = np.full(B, 140_000, dtype=np.int64)
        num_pages = int(sum(-(-int(x) // PAGE_TOKENS) for x in L))
        perm = rng.permutation(num_pages).astype(np.int32)
        table, _ = _pages_for(L, perm)
        topk = np.empty((B, Q, K), dtype=np.int64)
        for b in range(B):
            recent = _draw_without_replacement(rng, int(L[b]) - 4000, int(L[b]), K // 2)
            old = _draw_without_replacement(rng, 0, int(L[b]) - 4000, K - K // 2)
            topk[b, 0] = rng.permutation(np.concatenate([recent, old]))
        notes = {}
    elif cfg == 2:
        B, Q, H, K = 64, 1, 32, 2048
        L = rng.integers(70_000, 160_001, size=B).astype(np.int64)
        num_pages = int(sum(-(-int(x) // PAGE_TOKENS) for x in L))
        perm = rng.permutation(num_pages).astype(np.int32)
        table, _ = _pages_for(L, perm)
        topk = np.empty((B, Q, K), dtype=np.int64)
        for b in range(B):
            n = min(K, int(L[b]))
            sel = _draw_without_replacement(rng, 0, int(L[b]), n)
            topk[b, 0] = np.concatenate([sel, -np.ones(K - n, dtype=np.int64)])
        notes = {}
    elif cfg in (3, "3s"):
        B, Q, H, K = 32, 4, 32, 2048
        new_rows = 6000
        L_ctx = (rng.integers(100_000, 150_001, size=B) // PAGE_TOKENS) * PAGE_TOKENS
        L = L_ctx + new_rows
        num_pages = int(sum(-(-int(x) // PAGE_TOKENS) for x in L))
        perm = rng.permutation(num_pages).astype(np.int32)
        table, _ = _pages_for(L, perm)
        slots = []
        for b in range(B):
            pos = np.arange(int(L_ctx[b]), int(L[b]), dtype=np.int64)
            slots.append(table[b, pos // PAGE_TOKENS].astype(np.int64) * PAGE_TOKENS + pos % PAGE_TOKENS)
        topk = np.empty((B, Q, K), dtype=np.int64)
        for b in range(B):
            if cfg == "3s":
                topk[b] = _shared_lists(rng, int(L[b]), Q, K, SHARED_FRACTION)
                continue
            for j in range(Q):
                causal = int(L[b]) - Q + j       # last position query j may see
                topk[b, j] = _draw_without_replacement(rng, 0, causal + 1, K)
        notes = {"new_rows_per_request": new_rows, "L_ctx": L_ctx}
        if cfg == "3s":
            notes["shared_fraction"] = SHARED_FRACTION
        case_new_slots = np.concatenate(slots)
    elif cfg == 4:
        B, Q, H, K = 128, 1, 32, 2048
        num_pages = 25_469
        L = np.clip(np.round(rng.lognormal(math.log(12_000), 1.0, size=B)), 1000, 160_000).astype(np.int64)
        L[:4] = [1000, 1500, 2047, 2048]
        perm = rng.permutation(num_pages).astype(np.int32)
        table, used = _pages_for(L, perm, cycle=True)
        topk = np.empty((B, Q, K), dtype=np.int64)
        for b in range(B):
            n = min(K, int(L[b]))
            sel = _draw_without_replacement(rng, 0, int(L[b]), n)
            topk[b, 0] = np.concatenate([sel, -np.ones(K - n, dtype=np.int64)])
        notes = {"pages_referenced": used, "aliased_fraction": max(0.0, 1.0 - num_pages / used)}
    elif cfg == "4d":
        B, Q, H, K = 8, 1, 32, 8000
        L = np.full(B, 8000, dtype=np.int64)
        num_pages = int(sum(-(-int(x) // PAGE_TOKENS) for x in L))
        perm = rng.permutation(num_pages).astype(np.int32)
        table, _ = _pages_for(L, perm)
        topk = np.broadcast_to(np.arange(K, dtype=np.int64), (B, Q, K)).copy()
        notes = {"dense_control": True}
    else:
        raise ValueError(f"unknown config {cfg!r}")

    q_bits = _queries(rng, B, Q, H)
    case = DecodeCase(
        name=CONFIG_NAMES[cfg], B=B, Q=Q, H=H, topk=K, num_pages=num_pages,
        seq_lens=L.astype(np.int32), page_table=table, topk_indices=topk.astype(np.int32),
        q_bits=q_bits, channel_scale=c, row_seed=row_seed, notes=notes)
    if cfg in (3, "3s"):
        case.new_slots = case_new_slots
    return case


def small_case(B=2, Q=1, H=16, topk=200, L=(700, 1000), num_pages=None, seed=7,
               invalid_frac=0.0, dup=False, causal_tail=False, shared=None) -> DecodeCase:
    """A small random case for parity tests (a few tiles and a ragged tail).

    invalid_frac replaces that fraction of index entries with -1 or with
    positions past the sequence; causal_tail makes some entries point past the
    query's causal position; shared (a fraction) gives the Q tokens of a request
    lists that share that fraction of their positions (see _shared_lists).
    """
    rng = np.random.default_rng(seed)
    L = np.asarray(L, dtype=np.int64)
    assert L.size == B
    need = int(sum(-(-int(x) // PAGE_TOKENS) for x in L))
    if num_pages is None:
        num_pages = need + 3
    perm = rng.permutation(num_pages).astype(np.int32)
    table, _ = _pages_for(L, perm)
    topk = np.empty((B, Q, topk), dtype=np.int64)
    K = topk.shape[2]
    for b in range(B):
        shared_rows = None
        if shared is not None:
            assert int(L[b]) - Q + 1 >= 2 * K, "shared lists need a range of at least 2K positions"
            shared_rows = _shared_lists(rng, int(L[b]), Q, K, shared)
        for j in range(Q):
            hi = int(L[b]) - Q + j + 1
            n = min(K, hi)
            if shared_rows is not None:
                row = shared_rows[j].copy()
            else:
                sel = _draw_without_replacement(rng, 0, hi, n)
                row = np.concatenate([sel, -np.ones(K - n, dtype=np.int64)])
            if dup and n >= 2:
                row[1] = row[0]
            if invalid_frac > 0:
                m = rng.random(K) < invalid_frac
                kinds = rng.integers(0, 3, size=K)
                row = np.where(m & (kinds == 0), -1, row)
                row = np.where(m & (kinds == 1), int(L[b]) + rng.integers(0, 100, size=K), row)
                row = np.where(m & (kinds == 2), -2 - rng.integers(0, 5, size=K), row)
            if causal_tail and Q > 1:
                row[-1] = int(L[b]) - 1     # beyond the causal limit for j < Q-1
            topk[b, j] = row
    return DecodeCase(
        name=f"small B={B} Q={Q} H={H} K={K}", B=B, Q=Q, H=H, topk=K, num_pages=num_pages,
        seq_lens=L.astype(np.int32), page_table=table, topk_indices=topk.astype(np.int32),
        q_bits=_queries(rng, B, Q, H), channel_scale=_channel_scale(rng),
        row_seed=int(rng.integers(1, 2**31 - 1)))
