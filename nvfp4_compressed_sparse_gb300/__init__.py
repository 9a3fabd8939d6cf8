"""Python binding for libnvfp4mla (NVFP4-compressed paged MLA cache + sparse MLA decode).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libnvfp4mla.so. PyTorch is used for device memory and streams. If
the library cannot be loaded (or built with nvcc), importing the functions
raises; there is no CPU fallback.

C entry points (see include/nvfp4mla.h): mla_kv_pack,
sparse_mla_decode_workspace_size, sparse_mla_decode, sparse_mla_decode_plan,
sparse_mla_decode_noalloc, indexer_topk, fp8_kv_pack, nvfp4_stage_fp8,
sparse_mla_decode_fp8, fp8_token_kv_pack, sparse_mla_decode_fp8_token,
sparse_mla_decode_shared, nvfp4mla_status_string.
"""
from __future__ import annotations

import ctypes
import os
import threading

ROW_BYTES = 352
FP8_ROW_BYTES = 576
TOKEN_ROW_BYTES = 672
PAGE_TOKENS = 64
LATENT_DIM = 512
ROPE_DIM = 64
QK_DIM = 576
FLAG_TEST_TIMEOUT = 1 << 31   # NVFP4MLA_FLAG_TEST_TIMEOUT
FLAG_CLUSTER = 1 << 30        # NVFP4MLA_FLAG_CLUSTER
FLAG_CLUSTER_ANY = 1 << 29    # NVFP4MLA_FLAG_CLUSTER_ANY
FLAG_SPLIT = 1 << 28          # NVFP4MLA_FLAG_SPLIT
FLAG_PAIR = 1 << 27           # NVFP4MLA_FLAG_PAIR
STATUS_WORDS = 4
STAT_BAD_INDEX, STAT_BAD_PAGE, STAT_TIMEOUT, STAT_BAD_SLOT = 0, 1, 2, 3

_LIB = None
_LOCK = threading.Lock()


class NvFp4MlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


def lib_path() -> str:
    from . import _build
    return _build.LIB_PATH


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library; raise if impossible."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        from . import _build
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"libnvfp4mla.so not found at {_build.LIB_PATH}; build it with __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB_PATH)
        vp, i64, i32, u32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t
        lib.mla_kv_pack.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, vp]
        lib.mla_kv_pack.restype = i32
        lib.sparse_mla_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.sparse_mla_decode_workspace_size.restype = sz
        lib.sparse_mla_decode.argtypes = [vp, vp, i64, vp, i64, vp, vp, i32, i32, i32, i32, ctypes.c_float,
                                          vp, vp, vp, sz, vp, u32, vp]
        lib.sparse_mla_decode.restype = i32
        lib.sparse_mla_decode_plan.argtypes = [i32, i32, i32, i32, u32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.sparse_mla_decode_plan.restype = i32
        lib.indexer_topk.argtypes = [vp, i64, vp, i32, i32, i32, vp, vp]
        lib.indexer_topk.restype = i32
        lib.fp8_kv_pack.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, vp]
        lib.fp8_kv_pack.restype = i32
        lib.nvfp4_stage_fp8.argtypes = [vp, i64, vp, i64, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.nvfp4_stage_fp8.restype = i32
        lib.sparse_mla_decode_fp8.argtypes = [vp, vp, i64, vp, i64, vp, vp, i32, i32, i32, i32, ctypes.c_float,
                                              vp, vp, vp, sz, vp, vp]
        lib.sparse_mla_decode_fp8.restype = i32
        lib.sparse_mla_decode_shared.argtypes = [vp, vp, i64, vp, i64, vp, vp, vp, i32, i32, i32, i32,
                                                 ctypes.c_float, vp, vp, vp, sz, vp, u32, vp]
        lib.sparse_mla_decode_shared.restype = i32
        lib.fp8_token_kv_pack.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, vp]
        lib.fp8_token_kv_pack.restype = i32
        lib.sparse_mla_decode_fp8_token.argtypes = [vp, vp, i64, vp, i64, vp, vp, i32, i32, i32, i32, ctypes.c_float,
                                                    vp, vp, vp, sz, vp, vp]
        lib.sparse_mla_decode_fp8_token.restype = i32
        lib.nvfp4mla_status_string.argtypes = [i32]
        lib.nvfp4mla_status_string.restype = ctypes.c_char_p
        _LIB = lib
        return lib


def status_string(code: int) -> str:
    return load_library().nvfp4mla_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, device=None, ndim=None, contiguous=True, host_ok=False):
    """device: the CUDA device the tensor must be on. host_ok: a page-locked (pinned) CPU tensor
    is accepted too (the kernels read or write it over the host link)."""
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        if not (host_ok and t.device.type == "cpu" and t.is_pinned()):
            raise ValueError(f"{name}: must be a CUDA tensor" + (" or a pinned CPU tensor" if host_ok else ""))
    elif device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {t.dim()}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def mla_kv_pack(latent, rope, slot_mapping, kv_cache, dev_status=None, stream=None) -> None:
    """Encode bf16 latent [N,512] + rope [N,64] rows into kv_cache uint8 [P,64,352] at slot_mapping (int64 [N])."""
    import torch
    _check(latent, "latent", torch.bfloat16, ndim=2, contiguous=False)
    _check(rope, "rope", torch.bfloat16, latent.device, 2, contiguous=False)
    _check(slot_mapping, "slot_mapping", torch.int64, latent.device, 1)
    _check(kv_cache, "kv_cache", torch.uint8, latent.device, 3)
    if latent.stride(1) != 1 or rope.stride(1) != 1:
        raise ValueError("latent/rope rows must be contiguous along the feature axis")
    n = latent.shape[0]
    if latent.shape[1] != LATENT_DIM or rope.shape != (n, ROPE_DIM) or slot_mapping.shape[0] != n:
        raise ValueError("shape mismatch")
    if kv_cache.shape[1:] != (PAGE_TOKENS, ROW_BYTES):
        raise ValueError("kv_cache must be [num_pages, 64, 352]")
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, latent.device, 1)
    rc = load_library().mla_kv_pack(_ptr(latent), latent.stride(0), _ptr(rope), rope.stride(0), _ptr(slot_mapping),
                                    n, _ptr(kv_cache), kv_cache.shape[0], _ptr(dev_status), _stream_ptr(stream))
    if rc != 0:
        raise NvFp4MlaError(rc, "mla_kv_pack")


def indexer_topk(logits, seq_lens, topk: int, out=None, stream=None):
    """Top-k positions of each query's causal range from indexer logits fp32 [B, Q, S] (S a multiple
    of 4); seq_lens int32 [B]. Returns int32 [B, Q, topk] (increasing positions, -1 padded)."""
    import torch
    _check(logits, "logits", torch.float32, ndim=3)
    dev = logits.device
    _check(seq_lens, "seq_lens", torch.int32, dev, 1)
    B, Q, S = logits.shape
    if seq_lens.shape[0] != B:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, Q, topk), dtype=torch.int32, device=dev)
    _check(out, "out", torch.int32, dev, 3)
    if tuple(out.shape) != (B, Q, topk):
        raise ValueError("out must be [B, Q, topk]")
    rc = load_library().indexer_topk(_ptr(logits), S, _ptr(seq_lens), B, Q, topk, _ptr(out), _stream_ptr(stream))
    if rc != 0:
        raise NvFp4MlaError(rc, "indexer_topk")
    return out


def sparse_mla_decode_workspace_size(B: int, Q: int, H: int, topk: int, num_sms: int = 0) -> int:
    return int(load_library().sparse_mla_decode_workspace_size(B, Q, H, topk, num_sms))


def _cluster_flags(cluster) -> int:
    # cluster: None (the library's default schedule), False/"split" (always the split schedule),
    # True (also the cluster schedule wherever it is as balanced as the split one) or "any" (the
    # cluster schedule whenever one wave of clusters fits; a tuning aid) or "pair" (the split run by
    # 2-CTA clusters, one half of the contraction per CTA)
    if cluster is None:
        return 0
    if cluster is False or cluster == "split":
        return FLAG_SPLIT
    if cluster == "pair":
        return FLAG_PAIR
    return FLAG_CLUSTER | (FLAG_CLUSTER_ANY if cluster == "any" else 0)


def sparse_mla_decode_plan(B: int, Q: int, H: int, topk: int, max_ctas: int = 0,
                           cluster=None) -> tuple[int, int]:
    """(decode CTAs, cluster size G; 0 = split schedule, -2 = pair schedule) that sparse_mla_decode
    launches on the current device."""
    flags = (max_ctas & 0xFFFF) | _cluster_flags(cluster)
    ctas, g = ctypes.c_int(0), ctypes.c_int(0)
    rc = load_library().sparse_mla_decode_plan(B, Q, H, topk, flags, ctypes.byref(ctas), ctypes.byref(g))
    if rc != 0:
        raise NvFp4MlaError(rc, "sparse_mla_decode_plan")
    return ctas.value, g.value


def sparse_mla_decode(q, kv_cache, page_table, topk_indices, seq_lens, softmax_scale, out=None, lse=None,
                      workspace=None, dev_status=None, max_ctas: int = 0, stream=None,
                      test_timeout: bool = False, cluster=None):
    """One sparse MLA decode step. q bf16 [B,Q,H,576], kv_cache uint8 [P,64,352],
    page_table int32 [B,max_pages], topk_indices int32 [B,Q,K], seq_lens int32 [B].
    Returns (out bf16 [B,Q,H,512], lse fp32 [B,Q,H]). max_ctas and test_timeout are the
    testing aids NVFP4MLA_FLAG_MAX_CTAS and NVFP4MLA_FLAG_TEST_TIMEOUT; cluster=True sets
    NVFP4MLA_FLAG_CLUSTER (also the one-grid cluster schedule where it is as balanced as the
    split one; cluster="any" also sets NVFP4MLA_FLAG_CLUSTER_ANY), cluster=False sets
    NVFP4MLA_FLAG_SPLIT, None keeps the library's default. q, page_table, topk_indices,
    seq_lens, out and lse may be pinned CPU tensors: the kernels then read the inputs from and
    write the results to host memory directly, inside the call's stream order."""
    import torch
    _check(kv_cache, "kv_cache", torch.uint8, ndim=3)
    dev = kv_cache.device
    _check(q, "q", torch.bfloat16, dev, 4, host_ok=True)
    _check(page_table, "page_table", torch.int32, dev, 2, host_ok=True)
    _check(topk_indices, "topk_indices", torch.int32, dev, 3, host_ok=True)
    _check(seq_lens, "seq_lens", torch.int32, dev, 1, host_ok=True)
    B, Q, H, D = q.shape
    K = topk_indices.shape[2]
    if D != QK_DIM or topk_indices.shape[:2] != (B, Q) or seq_lens.shape[0] != B or page_table.shape[0] != B:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, Q, H, LATENT_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    _check(out, "out", torch.bfloat16, dev, 4, host_ok=True)
    _check(lse, "lse", torch.float32, dev, 3, host_ok=True)
    if workspace is None:
        nbytes = sparse_mla_decode_workspace_size(B, Q, H, K)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, dev, 1)
    rc = load_library().sparse_mla_decode(
        _ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(page_table), page_table.shape[1], _ptr(topk_indices),
        _ptr(seq_lens), B, Q, H, K, float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status),
        (int(max_ctas) & 0xFFFF) | (FLAG_TEST_TIMEOUT if test_timeout else 0) | _cluster_flags(cluster),
        _stream_ptr(stream))
    if rc != 0:
        raise NvFp4MlaError(rc, "sparse_mla_decode")
    return out, lse


# ------------------------------------------------------------------ FP8 comparison paths
def fp8_kv_pack(latent, rope, slot_mapping, kv_cache_fp8, dev_status=None, stream=None) -> None:
    """Encode bf16 latent [N,512] + rope [N,64] rows as 576-byte FP8 rows into kv_cache_fp8 uint8
    [P,64,576] at slot_mapping (int64 [N])."""
    _pack_rows("fp8_kv_pack", FP8_ROW_BYTES, latent, rope, slot_mapping, kv_cache_fp8, dev_status, stream)


def fp8_token_kv_pack(latent, rope, slot_mapping, kv_cache_tok, dev_status=None, stream=None) -> None:
    """Encode bf16 latent [N,512] + rope [N,64] rows as 672-byte per-token FP8 rows (E4M3 latent /
    scale, bf16 rope / scale, fp32 scale) into kv_cache_tok uint8 [P,64,672] at slot_mapping."""
    _pack_rows("fp8_token_kv_pack", TOKEN_ROW_BYTES, latent, rope, slot_mapping, kv_cache_tok, dev_status, stream)


def _pack_rows(entry, row_bytes, latent, rope, slot_mapping, kv_cache_fp8, dev_status, stream):
    import torch
    _check(latent, "latent", torch.bfloat16, ndim=2, contiguous=False)
    _check(rope, "rope", torch.bfloat16, latent.device, 2, contiguous=False)
    _check(slot_mapping, "slot_mapping", torch.int64, latent.device, 1)
    _check(kv_cache_fp8, "kv_cache_fp8", torch.uint8, latent.device, 3)
    if latent.stride(1) != 1 or rope.stride(1) != 1:
        raise ValueError("latent/rope rows must be contiguous along the feature axis")
    n = latent.shape[0]
    if latent.shape[1] != LATENT_DIM or rope.shape != (n, ROPE_DIM) or slot_mapping.shape[0] != n:
        raise ValueError("shape mismatch")
    if kv_cache_fp8.shape[1:] != (PAGE_TOKENS, row_bytes):
        raise ValueError(f"the cache must be [num_pages, 64, {row_bytes}]")
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, latent.device, 1)
    rc = getattr(load_library(), entry)(_ptr(latent), latent.stride(0), _ptr(rope), rope.stride(0),
                                        _ptr(slot_mapping), n, _ptr(kv_cache_fp8), kv_cache_fp8.shape[0],
                                        _ptr(dev_status), _stream_ptr(stream))
    if rc != 0:
        raise NvFp4MlaError(rc, entry)


def nvfp4_stage_fp8(kv_cache, page_table, topk_indices, seq_lens, staging=None, dev_status=None, stream=None):
    """The staging kernel of the staged path: FP8 copies of the selected NVFP4 rows of one decode
    step. Returns staging = (staged uint8 [B*Q*K/64, 64, 576], staged_indices int32 [B*Q, 1, K],
    staged_page_table int32 [B*Q, K/64], staged_seq_lens int32 [B*Q]), the cache, index lists,
    page table and lengths of sparse_mla_decode_fp8 over the staged rows (pass a previous result
    as staging to reuse its buffers)."""
    import torch
    _check(kv_cache, "kv_cache", torch.uint8, ndim=3)
    dev = kv_cache.device
    _check(page_table, "page_table", torch.int32, dev, 2)
    _check(topk_indices, "topk_indices", torch.int32, dev, 3)
    _check(seq_lens, "seq_lens", torch.int32, dev, 1)
    B, Q, K = topk_indices.shape
    if kv_cache.shape[1:] != (PAGE_TOKENS, ROW_BYTES) or seq_lens.shape[0] != B or page_table.shape[0] != B:
        raise ValueError("shape mismatch")
    if K % PAGE_TOKENS != 0:
        raise ValueError("topk must be a multiple of 64 for the staged path")
    U, P = B * Q, K // PAGE_TOKENS
    if staging is None:
        staging = (torch.empty((U * P, PAGE_TOKENS, FP8_ROW_BYTES), dtype=torch.uint8, device=dev),
                   torch.empty((U, 1, K), dtype=torch.int32, device=dev),
                   torch.empty((U, P), dtype=torch.int32, device=dev),
                   torch.empty((U,), dtype=torch.int32, device=dev))
    staged, sidx, spt, ssl = staging
    if (staged.shape != (U * P, PAGE_TOKENS, FP8_ROW_BYTES) or sidx.shape != (U, 1, K) or spt.shape != (U, P)
            or ssl.shape != (U,)):
        raise ValueError("staging buffers do not match the step's sizes")
    _check(staged, "staged", torch.uint8, dev)
    for t, name in ((sidx, "staged_indices"), (spt, "staged_page_table"), (ssl, "staged_seq_lens")):
        _check(t, name, torch.int32, dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, dev, 1)
    rc = load_library().nvfp4_stage_fp8(
        _ptr(kv_cache), kv_cache.shape[0], _ptr(page_table), page_table.shape[1], _ptr(topk_indices),
        _ptr(seq_lens), B, Q, K, _ptr(staged), _ptr(sidx), _ptr(spt), _ptr(ssl), _ptr(dev_status),
        _stream_ptr(stream))
    if rc != 0:
        raise NvFp4MlaError(rc, "nvfp4_stage_fp8")
    return staging


def sparse_mla_decode_fp8(q, kv_cache_fp8, page_table, topk_indices, seq_lens, softmax_scale, out=None, lse=None,
                          workspace=None, dev_status=None, stream=None):
    """sparse_mla_decode over a cache of 576-byte FP8 rows (uint8 [P,64,576]); device tensors only."""
    return _decode_rows("sparse_mla_decode_fp8", FP8_ROW_BYTES, q, kv_cache_fp8, page_table, topk_indices, seq_lens,
                        softmax_scale, out, lse, workspace, dev_status, stream)


def sparse_mla_decode_fp8_token(q, kv_cache_tok, page_table, topk_indices, seq_lens, softmax_scale, out=None,
                                lse=None, workspace=None, dev_status=None, stream=None):
    """sparse_mla_decode over a cache of 672-byte per-token FP8 rows (uint8 [P,64,672]); device tensors only."""
    return _decode_rows("sparse_mla_decode_fp8_token", TOKEN_ROW_BYTES, q, kv_cache_tok, page_table, topk_indices,
                        seq_lens, softmax_scale, out, lse, workspace, dev_status, stream)


def _decode_rows(entry, row_bytes, q, kv_cache_fp8, page_table, topk_indices, seq_lens, softmax_scale, out, lse,
                 workspace, dev_status, stream):
    import torch
    _check(kv_cache_fp8, "kv_cache", torch.uint8, ndim=3)
    dev = kv_cache_fp8.device
    if kv_cache_fp8.shape[1:] != (PAGE_TOKENS, row_bytes):
        raise ValueError(f"the cache must be [num_pages, 64, {row_bytes}]")
    _check(q, "q", torch.bfloat16, dev, 4)
    _check(page_table, "page_table", torch.int32, dev, 2)
    _check(topk_indices, "topk_indices", torch.int32, dev, 3)
    _check(seq_lens, "seq_lens", torch.int32, dev, 1)
    B, Q, H, D = q.shape
    K = topk_indices.shape[2]
    if D != QK_DIM or topk_indices.shape[:2] != (B, Q) or seq_lens.shape[0] != B or page_table.shape[0] != B:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, Q, H, LATENT_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    _check(out, "out", torch.bfloat16, dev, 4)
    _check(lse, "lse", torch.float32, dev, 3)
    if workspace is None:
        workspace = torch.empty(max(sparse_mla_decode_workspace_size(B, Q, H, K), 1), dtype=torch.uint8, device=dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, dev, 1)
    rc = getattr(load_library(), entry)(
        _ptr(q), _ptr(kv_cache_fp8), kv_cache_fp8.shape[0], _ptr(page_table), page_table.shape[1],
        _ptr(topk_indices), _ptr(seq_lens), B, Q, H, K, float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream_ptr(stream))
    if rc != 0:
        raise NvFp4MlaError(rc, entry)
    return out, lse


def staged_sparse_mla_decode(q, kv_cache, page_table, topk_indices, seq_lens, softmax_scale, staging=None,
                             out=None, lse=None, workspace=None, dev_status=None, stream=None):
    """The staged path of one decode step: nvfp4_stage_fp8, then sparse_mla_decode_fp8 over the
    staged rows as B*Q one-query requests. Same inputs and outputs as sparse_mla_decode (device
    tensors). Returns (out, lse, staging)."""
    B, Q, H, _ = q.shape
    staging = nvfp4_stage_fp8(kv_cache, page_table, topk_indices, seq_lens, staging, dev_status, stream)
    staged, sidx, spt, ssl = staging
    o = None if out is None else out.view(B * Q, 1, H, LATENT_DIM)
    s = None if lse is None else lse.view(B * Q, 1, H)
    o, s = sparse_mla_decode_fp8(q.reshape(B * Q, 1, H, QK_DIM), staged, spt, sidx, ssl, softmax_scale, o, s,
                                 workspace, dev_status, stream)
    return o.view(B, Q, H, LATENT_DIM), s.view(B, Q, H), staging


def sparse_mla_decode_shared(q, kv_cache, page_table, shared_indices, member_masks, seq_lens, softmax_scale,
                             out=None, lse=None, workspace=None, dev_status=None, stream=None, cluster=None):
    """The Q query tokens of each request folded over one shared index list: q bf16 [B,Q,H,576],
    shared_indices int32 [B,K], member_masks uint8 [B,K] (bit j: entry in query j's list).
    Returns (out bf16 [B,Q,H,512], lse fp32 [B,Q,H]). Always the split schedule (cluster flags
    are ignored); device tensors only."""
    import torch
    _check(kv_cache, "kv_cache", torch.uint8, ndim=3)
    dev = kv_cache.device
    _check(q, "q", torch.bfloat16, dev, 4)
    _check(page_table, "page_table", torch.int32, dev, 2)
    _check(shared_indices, "shared_indices", torch.int32, dev, 2)
    _check(member_masks, "member_masks", torch.uint8, dev, 2)
    _check(seq_lens, "seq_lens", torch.int32, dev, 1)
    B, Q, H, D = q.shape
    K = shared_indices.shape[1]
    if (D != QK_DIM or shared_indices.shape[0] != B or tuple(member_masks.shape) != (B, K) or seq_lens.shape[0] != B
            or page_table.shape[0] != B):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, Q, H, LATENT_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    _check(out, "out", torch.bfloat16, dev, 4)
    _check(lse, "lse", torch.float32, dev, 3)
    if workspace is None:
        workspace = torch.empty(max(sparse_mla_decode_workspace_size(B, 1, Q * H, K), 1), dtype=torch.uint8,
                                device=dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, dev, 1)
    rc = load_library().sparse_mla_decode_shared(
        _ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(page_table), page_table.shape[1], _ptr(shared_indices),
        _ptr(member_masks), _ptr(seq_lens), B, Q, H, K, float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _cluster_flags(cluster), _stream_ptr(stream))
    if rc != 0:
        raise NvFp4MlaError(rc, "sparse_mla_decode_shared")
    return out, lse
