"""mla_kv_pack on the GPU vs the CPU oracle: bit-exact cache bytes."""
import numpy as np
import pytest
import torch

import nvfp4_compressed_sparse_gb300 as m
import workloads
from oracle import codec, pack
from tests.gpu_util import bf16_dev, bits_of

pytestmark = pytest.mark.gpu


def _finite_bf16():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    return b[((b >> 7) & 0xFF) != 0xFF]


def _run_pack(lat_bits, rope_bits, slots, num_pages, fill=0xCD, status=None):
    cache = torch.full((num_pages, 64, 352), fill, dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(bf16_dev(lat_bits), bf16_dev(rope_bits), torch.from_numpy(np.asarray(slots, np.int64)).cuda(),
                  cache, dev_status=status)
    torch.cuda.synchronize()
    return cache.cpu().numpy()


def _check_rows(lat_bits, rope_bits):
    n = lat_bits.shape[0]
    pages = -(-n // 64)
    got = _run_pack(lat_bits, rope_bits, np.arange(n), pages).reshape(-1, 352)[:n]
    want = pack.encode_rows(lat_bits, rope_bits)
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:5]}"


def test_random_rows_with_sentinels():
    case = workloads.small_case(B=1, Q=1, H=16, topk=10, L=(640,), num_pages=12, seed=5)
    lat, rope = workloads.host_rows(case, np.arange(12))
    rng = np.random.default_rng(0)
    slots = rng.permutation(12 * 64)[:500].astype(np.int64)
    slots[::17] = -1
    got = _run_pack(lat[:500], rope[:500], slots, 12)
    want = np.full((12, 64, 352), 0xCD, np.uint8)
    pack.write_cache(want, lat[:500], rope[:500], slots)
    np.testing.assert_array_equal(got, want)


def test_scale_of_every_bf16_amax():
    bits = _finite_bf16()
    bits = bits[bits < 0x8000]
    n_blocks = -(-bits.size // 32) * 32
    lat = np.zeros((n_blocks, 16), np.uint16)
    lat[:bits.size, 0] = bits
    lat[:bits.size, 1] = bits | 0x8000          # the same magnitude, negative
    _check_rows(lat.reshape(-1, 512), np.zeros((n_blocks // 32, 64), np.uint16))


def test_every_value_under_every_scale():
    """For each of the 126 positive E4M3 scales s: blocks with amax = 6s whose other
    15 entries run through every bf16 value of magnitude <= 6s (both signs)."""
    allb = _finite_bf16()
    vals = codec.bf16_bits_to_f64(allb)
    blocks = []
    for s in codec.e4m3_decode(np.arange(1, 0x7F)):
        amax_bits = workloads.f32_to_bf16_bits(np.array([6 * s], np.float32))[0]
        sel = allb[np.abs(vals) <= 6 * s]
        k = -(-sel.size // 15) * 15
        fill = np.resize(sel, k).reshape(-1, 15)
        blk = np.concatenate([np.full((fill.shape[0], 1), amax_bits, np.uint16), fill], axis=1)
        blocks.append(blk)
    blocks = np.concatenate(blocks)
    blocks = np.concatenate([blocks, np.zeros((-blocks.shape[0] % 32, 16), np.uint16)])
    lat = blocks.reshape(-1, 512)
    _check_rows(lat, np.zeros((lat.shape[0], 64), np.uint16))


def test_rope_every_bf16():
    bits = _finite_bf16()
    n = -(-bits.size // 64) * 64
    rope = np.zeros(n, np.uint16)
    rope[:bits.size] = bits
    rope = rope.reshape(-1, 64)
    _check_rows(np.zeros((rope.shape[0], 512), np.uint16), rope)


def test_bad_slots_are_skipped_and_counted():
    case = workloads.small_case(B=1, Q=1, H=16, topk=10, L=(64,), num_pages=2, seed=1)
    lat, rope = workloads.host_rows(case, np.arange(1))
    slots = np.array([0, -1, 128, -7, 5, 10**12] + list(range(20, 78)), np.int64)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    got = _run_pack(lat, rope, slots, 2, status=status)
    want = np.full((2, 64, 352), 0xCD, np.uint8)
    res = pack.write_cache(want, lat, rope, slots)
    np.testing.assert_array_equal(got, want)
    assert status.cpu().tolist() == [0, 0, 0, res["bad_slots"]] and res["bad_slots"] == 3


def test_strided_rows():
    case = workloads.small_case(B=1, Q=1, H=16, topk=10, L=(128,), num_pages=2, seed=2)
    lat, rope = workloads.host_rows(case, np.arange(2))
    big = torch.zeros((128, 600), dtype=torch.bfloat16, device="cuda")
    big[:, :512] = bf16_dev(lat)
    bigr = torch.zeros((128, 80), dtype=torch.bfloat16, device="cuda")
    bigr[:, 8:72] = bf16_dev(rope)
    cache = torch.zeros((2, 64, 352), dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(big[:, :512], bigr[:, 8:72], torch.arange(128, device="cuda"), cache)
    np.testing.assert_array_equal(cache.cpu().numpy().reshape(-1, 352), pack.encode_rows(lat, rope))


def test_empty_pack_is_noop():
    cache = torch.full((1, 64, 352), 7, dtype=torch.uint8, device="cuda")
    m.mla_kv_pack(torch.zeros((0, 512), dtype=torch.bfloat16, device="cuda"),
                  torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"),
                  torch.zeros(0, dtype=torch.int64, device="cuda"), cache)
    assert (cache == 7).all()


def test_spec_verify_append_full_size_sampled():
    """The spec-verify case's 6,000-row-per-request append (192,000 rows) into fresh
    pages, in the bench's launch configuration; sampled rows bit-exact and no other
    row touched."""
    case = workloads.make_case(3)
    n = case.new_slots.size
    lat, rope = workloads.device_rows(case, n, "cuda", seed_offset=7)
    cache = torch.full((case.num_pages, 64, 352), 0xCD, dtype=torch.uint8, device="cuda")
    slots = torch.from_numpy(case.new_slots).cuda()
    m.mla_kv_pack(lat, rope, slots, cache)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    pick = rng.choice(n, 3000, replace=False)
    pt = torch.from_numpy(pick).cuda()
    want = pack.encode_rows(bits_of(lat[pt]), bits_of(rope[pt]))
    flat = cache.view(-1, 352)
    got = flat[slots[pt]].cpu().numpy()
    np.testing.assert_array_equal(got, want)
    written = torch.zeros(flat.shape[0], dtype=torch.bool, device="cuda")
    written[slots] = True
    assert bool((flat[~written] == 0xCD).all())


def test_non_finite_latent_and_rope_bit_exact():
    """NaN (both signs, several payloads) and +-inf in latent blocks and rope values: the kernel's
    bytes equal the oracle's under the stated reading (NaN out of the block maximum, coded as a
    signed zero; infinity saturating; rope NaN -> E4M3 NaN with sign, rope inf -> +-448)."""
    rng = np.random.default_rng(11)
    specials = np.array([0x7FC0, 0xFFC0, 0x7F81, 0xFFFF, 0x7F80, 0xFF80], np.uint16)
    n = 256
    lat = workloads.f32_to_bf16_bits(rng.standard_normal((n, 512), dtype=np.float32))
    rope = workloads.f32_to_bf16_bits(rng.standard_normal((n, 64), dtype=np.float32))
    # each row gets specials in a few random positions; some blocks are all NaN
    for r in range(n):
        k = int(rng.integers(1, 6))
        lat[r, rng.integers(0, 512, size=k)] = specials[rng.integers(0, specials.size, size=k)]
        rope[r, rng.integers(0, 64, size=2)] = specials[rng.integers(0, specials.size, size=2)]
    lat[0, 0:16] = 0x7FC0
    lat[1, 16:32] = np.where(np.arange(16) % 2 == 0, 0xFFC0, 0)
    lat[2, 32:48] = 0x7F80
    with np.errstate(all="ignore"):
        _check_rows(lat, rope)


def test_host_memory_rejected_before_launch():
    """Device inputs but a host-memory cache (pageable, then page-locked): the call returns
    INVALID_ARG before launching, and the cache bytes are untouched."""
    import ctypes
    lib = m.load_library()
    V = ctypes.c_void_p
    lat = torch.zeros((64, 512), dtype=torch.bfloat16, device="cuda")
    rope = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    slots = torch.arange(64, device="cuda")
    for pinned in (False, True):
        cache = torch.full((1, 64, 352), 0xAB, dtype=torch.uint8)
        if pinned:
            cache = cache.pin_memory()
        rc = lib.mla_kv_pack(V(lat.data_ptr()), 512, V(rope.data_ptr()), 64, V(slots.data_ptr()), 64,
                             V(cache.data_ptr()), 1, None, None)
        torch.cuda.synchronize()
        assert rc == 1, (pinned, rc)
        assert bool((cache == 0xAB).all())
    with pytest.raises(ValueError):
        m.mla_kv_pack(lat.cpu(), rope, slots, torch.zeros((1, 64, 352), dtype=torch.uint8, device="cuda"))
