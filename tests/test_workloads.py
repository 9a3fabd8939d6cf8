"""The seeded generators produce the shapes and structure the cases promise (CPU)."""
import numpy as np
import pytest

import workloads


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4, "4d"])
def test_case_structure(cfg):
    c = workloads.make_case(cfg)
    assert c.q_bits.shape == (c.B, c.Q, c.H, 576) and c.q_bits.dtype == np.uint16
    assert c.topk_indices.shape == (c.B, c.Q, c.topk)
    assert c.seq_lens.shape == (c.B,)
    for b in range(c.B):
        L = int(c.seq_lens[b])
        need = -(-L // 64)
        assert (c.page_table[b, :need] >= 0).all() and (c.page_table[b, :need] < c.num_pages).all()
        for j in range(c.Q):
            row = c.topk_indices[b, j]
            valid = row[row >= 0]
            assert valid.size == min(c.topk, L - c.Q + j + 1)
            assert np.unique(valid).size == valid.size
            assert (valid <= L - c.Q + j).all()
            assert (row[valid.size:] == -1).all() if valid.size < c.topk else True
    if cfg not in (4,):
        used = np.concatenate([c.page_table[b, :-(-int(c.seq_lens[b]) // 64)] for b in range(c.B)])
        assert np.unique(used).size == used.size       # no sharing outside the capacity case
    if cfg == 3:
        assert c.new_slots.size == 32 * 6000 and np.unique(c.new_slots).size == c.new_slots.size
    if cfg == 4:
        assert c.num_pages * 64 == 1_630_016
        assert c.seq_lens[:4].tolist() == [1000, 1500, 2047, 2048]
        assert c.notes["aliased_fraction"] > 0


def test_deterministic():
    a, b = workloads.make_case(2), workloads.make_case(2)
    np.testing.assert_array_equal(a.topk_indices, b.topk_indices)
    np.testing.assert_array_equal(a.q_bits, b.q_bits)
    ra = workloads.host_rows(a, [5, 9])
    rb = workloads.host_rows(b, [5, 9])
    np.testing.assert_array_equal(ra[0], rb[0])
    # a page's rows do not depend on which other pages are drawn with it
    np.testing.assert_array_equal(workloads.host_rows(a, [9])[0], ra[0][64:])


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 0.0, -0.0], np.float32)
    bits = workloads.f32_to_bf16_bits(x)
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000, 0x8000]


def test_fold_lists_round_trip():
    """The shared list and member bits give back each query's set of entries (duplicates merged)."""
    rng = np.random.default_rng(0)
    lists = rng.integers(-1, 50, size=(3, 4, 20))
    shared, member = workloads.fold_lists(lists)
    for b in range(3):
        for j in range(4):
            got = set(shared[b][((member[b] >> j) & 1).astype(bool)].tolist())
            assert got == set(lists[b, j].tolist()) - {-1}
        u = shared[b][shared[b] != -1]
        assert (np.diff(u) > 0).all() and not member[b][shared[b] == -1].any()


def test_subset_and_shared_lists_shapes():
    rng = np.random.default_rng(1)
    L, Q, K = 9000, 4, 512
    sub = workloads.subset_lists(rng, L, Q, K, 0.9)
    assert sub.shape == (Q, K) and all((sub[j] != -1).sum() == round(0.9 * K) for j in range(Q))
    assert np.unique(sub[sub != -1]).size <= K and sub.max() <= L - Q
    sh = workloads._shared_lists(rng, L, Q, K, 0.9)
    for j in range(Q):
        assert np.unique(sh[j]).size == K and sh[j].max() <= L - Q + j and (np.diff(sh[j]) > 0).all()
