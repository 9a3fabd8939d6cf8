"""The pack kernel forms a block's scale as E4M3_rn_sat(amax * RN32(1/6)) instead of dividing by
6. Here, on the CPU, that product (an IEEE binary32 multiply, as the kernel's) is checked against
the oracle's E4M3 rounding of the quotient amax / 6 for every non-negative bf16 amax, +inf
included. ("Serving GLM-5.3 ...", "Four bits per latent value": one E4M3 scale per 16 values;
the divisor 6 is the largest e2m1 magnitude.)"""
import numpy as np

from oracle import codec


def test_reciprocal_product_rounds_like_the_quotient():
    bits = np.arange(0, 0x7F81, dtype=np.uint32)          # +0 .. +inf as bf16 patterns
    amax = (bits << 16).view(np.float32)
    rcp6 = np.uint32(0x3E2AAAAB).view(np.float32)
    assert rcp6 == np.float32(1.0) / np.float32(6.0)      # RN32(1/6)
    product = amax * rcp6                                  # binary32, round to nearest
    want = codec.e4m3_encode(amax.astype(np.float64) / 6.0)
    got = codec.e4m3_encode(product.astype(np.float64))
    np.testing.assert_array_equal(got, want)
    # the ties of E4M3 rounding are among the inputs (amax = 6 x a midpoint): e.g. 6 x 2^-10,
    # which must round to 0 (even), and 6 x 17/16 (between 1 and 1.125), which must round to 1
    for a, code in [(6 * 2.0 ** -10, 0x00), (6 * 17 / 16, 0x38)]:
        a32 = np.float32(a)
        assert float(a32) == a
        assert codec.e4m3_encode(np.float64(a32 * rcp6)) == code
