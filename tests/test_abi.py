"""The C-ABI library builds, loads and exports every symbol its header declares;
host-side argument checks return the documented codes (CPU only: no call here
reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

import nvfp4_compressed_sparse_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4mla.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?[\s\*]+([A-Za-z_][A-Za-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


@pytest.fixture(scope="module")
def lib():
    return m.load_library()


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(names) >= {"mla_kv_pack", "sparse_mla_decode", "sparse_mla_decode_workspace_size",
                          "sparse_mla_decode_plan", "sparse_mla_decode_noalloc", "indexer_topk", "fp8_kv_pack",
                          "nvfp4_stage_fp8", "sparse_mla_decode_fp8", "fp8_token_kv_pack",
                          "sparse_mla_decode_fp8_token", "nvfp4mla_status_string"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert m.status_string(0) == "ok"
    for code in range(1, 6):
        assert m.status_string(code) not in ("ok", "unknown status")
    assert m.status_string(99) == "unknown status"


def _ws(slots, units, nh):
    r = lambda x: (x + 255) // 256 * 256
    return r(slots * nh * 512 * 4) + r(slots * nh * 2 * 4) + r(units * 9 * nh * 128) + r(units * 4) + r(slots * 8)


def test_workspace_size_formula(lib):
    # 152 SMs, B=64, Q=1, H=32, topk=2048: 64 units x 16 tiles; 152 CTAs; 215 partial slots
    assert lib.sparse_mla_decode_workspace_size(64, 1, 32, 2048, 152) == _ws(152 + 64 - 1, 64, 32)
    # fewer tiles than SMs: one CTA per tile
    assert lib.sparse_mla_decode_workspace_size(1, 1, 16, 256, 152) == _ws(2 + 1 - 1, 1, 16)
    # H=128 -> 4 head groups of 32
    assert lib.sparse_mla_decode_workspace_size(2, 1, 128, 128, 152) == _ws(8 + 8 - 1, 8, 32)
    for bad in [(0, 1, 32, 2048), (1, 0, 32, 2048), (1, 17, 32, 2048), (1, 1, 48, 2048), (1, 1, 32, 0), (1, 1, 32, 8193)]:
        assert lib.sparse_mla_decode_workspace_size(*bad, 152) == 0


V = ctypes.c_void_p


def _pack(lib, lat=16, lstride=512, rope=16, rstride=64, slots=8, n=1, cache=16, pages=1, status=None):
    return lib.mla_kv_pack(V(lat), lstride, V(rope), rstride, V(slots), n, V(cache), pages,
                           V(status) if status else None, None)


def test_pack_host_checks(lib):
    A = 1 << 20     # a fake, well aligned address (never dereferenced: every call fails its checks or n == 0)
    assert _pack(lib, A, n=0) == 0
    assert _pack(lib, A, n=-1) == 1
    assert _pack(lib, 0, rope=A, slots=A, cache=A) == 1
    assert _pack(lib, A, rope=0, slots=A, cache=A) == 1
    assert _pack(lib, A, rope=A, slots=0, cache=A) == 1
    assert _pack(lib, A, rope=A, slots=A, cache=0) == 1
    assert _pack(lib, A, rope=A, slots=A, cache=A, pages=0) == 1
    assert _pack(lib, A, lstride=500, rope=A, slots=A, cache=A) == 1
    assert _pack(lib, A + 8, rope=A, slots=A, cache=A) == 2
    assert _pack(lib, A, lstride=516, rope=A, slots=A, cache=A) == 2
    assert _pack(lib, A, rope=A + 2, slots=A, cache=A) == 2
    assert _pack(lib, A, rope=A, rstride=65, slots=A, cache=A) == 2
    assert _pack(lib, A, rope=A, slots=A + 4, cache=A) == 2
    assert _pack(lib, A, rope=A, slots=A, cache=A + 8) == 2


def test_pack_rejects_host_memory_before_launch(lib):
    """Real host buffers (pageable numpy memory), correctly sized and aligned: the pack call
    classifies its pointers first and returns INVALID_ARG without touching the cache."""
    import numpy as np
    lat = np.zeros((4, 512), np.uint16)
    rope = np.zeros((4, 64), np.uint16)
    slots = np.arange(4, dtype=np.int64)
    cache = np.full((1, 64, 352), 0xAB, np.uint8)
    P = lambda a: V(a.ctypes.data)
    rc = lib.mla_kv_pack(P(lat), 512, P(rope), 64, P(slots), 4, P(cache), 1, None, None)
    assert rc == 1
    assert (cache == 0xAB).all()


def _dec(lib, q=1 << 20, cache=1 << 20, pages=10, pt=1 << 20, maxp=4, idx=1 << 20, sl=1 << 20, B=1, Q=1, H=32,
         K=128, scale=0.07, out=1 << 20, lse=1 << 20, ws=1 << 20, wsb=1 << 30, status=None, flags=0):
    return lib.sparse_mla_decode(V(q), V(cache), pages, V(pt), maxp, V(idx), V(sl), B, Q, H, K, ctypes.c_float(scale),
                                 V(out), V(lse), V(ws), wsb, V(status) if status else None, flags, None)


def test_decode_host_checks(lib):
    A = 1 << 20
    for kw in [dict(B=0), dict(Q=0), dict(Q=17), dict(H=8), dict(H=48), dict(K=0), dict(K=9000), dict(q=0),
               dict(cache=0), dict(pt=0), dict(idx=0), dict(sl=0), dict(out=0), dict(lse=0), dict(pages=0),
               dict(maxp=0), dict(scale=0.0), dict(scale=-1.0), dict(scale=float("nan"))]:
        assert _dec(lib, **kw) == 1, kw
    for kw in [dict(q=A + 8), dict(cache=A + 4), dict(out=A + 2), dict(pt=A + 2), dict(idx=A + 1), dict(sl=A + 2),
               dict(lse=A + 2)]:
        assert _dec(lib, **kw) == 2, kw


def test_comparison_path_host_checks(lib):
    """The FP8 packs, the staging, the FP8 decodes and top-k reject bad sizes, NULLs, misalignment
    and host memory before any launch (these calls never reach a kernel here)."""
    import numpy as np
    A = 1 << 20
    for entry in (lib.fp8_kv_pack, lib.fp8_token_kv_pack):
        assert entry(V(A), 512, V(A), 64, V(A), 4, V(A), 0, None, None) == 1          # no pages
        assert entry(V(A), 511, V(A), 64, V(A), 4, V(A), 1, None, None) == 1          # row stride too small
        assert entry(V(A + 8), 512, V(A), 64, V(A), 4, V(A), 1, None, None) == 2      # latent not 16-byte aligned
        assert entry(None, 512, V(A), 64, V(A), 4, V(A), 1, None, None) == 1
        lat, rope = np.zeros((4, 512), np.uint16), np.zeros((4, 64), np.uint16)
        slots, cache = np.arange(4, dtype=np.int64), np.full((1, 64, 672), 0xAB, np.uint8)
        Pn = lambda a: V(a.ctypes.data)
        assert entry(Pn(lat), 512, Pn(rope), 64, Pn(slots), 4, Pn(cache), 1, None, None) == 1   # host memory
        assert (cache == 0xAB).all()
    st = lambda **kw: lib.nvfp4_stage_fp8(V(kw.get("cache", A)), 10, V(A), 4, V(A), V(A), kw.get("B", 1), 1,
                                          kw.get("K", 128), V(kw.get("staged", A)), V(A), V(A), V(A), None, None)
    assert st(K=100) == 1                                                              # not a multiple of 64
    assert st(K=0) == 1 and st(B=0) == 1
    assert st(staged=A + 4) == 2
    for entry in (lib.sparse_mla_decode_fp8, lib.sparse_mla_decode_fp8_token):
        assert entry(V(A), V(A), 10, V(A), 4, V(A), V(A), 1, 1, 32, 0, ctypes.c_float(0.07), V(A), V(A), V(A),
                     1 << 30, None, None) == 1                                         # topk 0
        assert entry(V(A), V(A), 10, V(A), 4, V(A), V(A), 1, 1, 48, 128, ctypes.c_float(0.07), V(A), V(A), V(A),
                     1 << 30, None, None) == 1                                         # H not supported
    tk = lambda **kw: lib.indexer_topk(V(kw.get("lg", A)), kw.get("S", 64), V(A), kw.get("B", 1), kw.get("Q", 1),
                                       kw.get("K", 8), V(A), None)
    assert tk(B=0) == 1 and tk(Q=17) == 1 and tk(K=0) == 1 and tk(K=9000) == 1 and tk(S=0) == 1
    assert tk(S=62) == 2 and tk(lg=A + 4) == 2


def test_binding_flag_constants_match_the_header():
    """The binding's schedule and testing flags are the header's bit values."""
    text = open(os.path.join(ROOT, "include", "nvfp4mla.h")).read()
    found = dict(re.findall(r"#define NVFP4MLA_FLAG_(\w+) \(1u << (\d+)\)", text))
    assert set(found) == {"TEST_TIMEOUT", "CLUSTER", "CLUSTER_ANY", "SPLIT", "PAIR"}
    for name, bit in found.items():
        assert getattr(m, "FLAG_" + name) == 1 << int(bit), name
