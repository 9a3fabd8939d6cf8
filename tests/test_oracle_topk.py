"""Pins for the oracle's top-k selection (CPU only): brute force with Python's own sort on the
stated rule, the key order against float comparison, and the special cases of the rule."""
import random
import struct

import numpy as np

from oracle import topk


def _brute(row, n, K):
    """Python sort on (value, position) with the rule written out directly."""
    def rank(i):
        v = float(row[i])
        if v != v:                       # NaN below every number
            return (0, 0.0, 0, -i)
        sign_bit = struct.unpack("<I", struct.pack("<f", row[i]))[0] >> 31
        return (1, v, 0 if sign_bit else 1, -i)   # -0.0 below +0.0, then smaller position first
    cand = sorted(range(min(n, len(row))), key=rank, reverse=True)[:K]
    out = sorted(cand) + [-1] * (K - len(cand))
    return np.array(out, dtype=np.int32)


def test_keys_order_like_floats():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 5000),
                        np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.4e38, -3.4e38], np.float32)])
    k = topk.order_keys(x).astype(np.int64)
    i, j = rng.integers(0, x.size, 20000), rng.integers(0, x.size, 20000)
    strict = x[i] < x[j]
    assert np.all(k[i][strict] < k[j][strict])
    equal_nonzero = (x[i] == x[j]) & (x[i] != 0)
    assert np.all(k[i][equal_nonzero] == k[j][equal_nonzero])
    assert topk.order_keys(np.array([-0.0], np.float32))[0] < topk.order_keys(np.array([0.0], np.float32))[0]
    nan = topk.order_keys(np.array([np.nan, -np.nan, -np.inf], np.float32))
    assert nan[0] == 0 and nan[1] == 0 and nan[2] > 0


def test_against_brute_force_with_ties_nan_and_short_rows():
    rng = np.random.default_rng(1)
    for trial in range(300):
        S = int(rng.integers(1, 200))
        K = int(rng.integers(1, 64))
        n = int(rng.integers(0, S + 5))
        row = rng.standard_normal(S).astype(np.float32)
        if trial % 3 == 0:
            row = np.round(row * 2) / 2                      # many ties
        if trial % 5 == 0:
            row[rng.integers(0, S, size=max(1, S // 10))] = np.nan
        if trial % 7 == 0:
            row[rng.integers(0, S, size=max(1, S // 10))] = -0.0
        np.testing.assert_array_equal(topk.select_row(row, n, K), _brute(row, n, K), err_msg=f"trial {trial}")


def test_special_cases():
    row = np.full(100, 3.0, np.float32)
    np.testing.assert_array_equal(topk.select_row(row, 100, 10), np.arange(10))        # all equal: first K
    np.testing.assert_array_equal(topk.select_row(row, 5, 8), [0, 1, 2, 3, 4, -1, -1, -1])
    np.testing.assert_array_equal(topk.select_row(row, 0, 3), [-1, -1, -1])
    row = np.arange(50, dtype=np.float32)
    np.testing.assert_array_equal(topk.select_row(row, 50, 5), [45, 46, 47, 48, 49])
    np.testing.assert_array_equal(topk.select_row(row, 30, 5), [25, 26, 27, 28, 29])   # causal range cut
    # the selected set does not depend on where the values sit, only on the values and ties
    rng = np.random.default_rng(3)
    v = rng.permutation(1000).astype(np.float32)
    perm = rng.permutation(1000)
    sel = topk.select_row(v, 1000, 100)
    sel_p = topk.select_row(v[perm], 1000, 100)
    assert sorted(v[sel].tolist()) == sorted(v[perm][sel_p].tolist()) == list(range(900, 1000))


def test_batch_causal_ranges():
    rng = np.random.default_rng(4)
    B, Q, S, K = 3, 4, 300, 50
    logits = rng.standard_normal((B, Q, S)).astype(np.float32)
    L = np.array([300, 120, 40])
    out = topk.select(logits, L, Q, K)
    for b in range(B):
        for j in range(Q):
            n = L[b] - Q + j + 1
            np.testing.assert_array_equal(out[b, j], _brute(logits[b, j], n, K))
            assert (out[b, j][out[b, j] >= 0] < n).all()
