"""The hidden-state projection runs on the tensor cores with h split into three bf16 terms:
h0 = bf16(h), h1 = bf16(h - h0), h2 = bf16(h - h0 - h1), each rounded to nearest even.
Its fp32 accuracy rests on two facts checked here with numpy, independently of the
kernel: the split is exact (h0 + h1 + h2 == h for every finite fp32 h with |h| >= 2^-110,
so that the remainders stay normal numbers; hidden states are far above that), and every
bf16 x bf16 product is exact in fp32 (8 + 8 significant bits).
"""
import numpy as np


def bf16_rne(x):
    """float32 array -> float32 values rounded to bf16 (round to nearest, ties to even)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (r.astype(np.uint32) << 16).view(np.float32)


def split3(h):
    h = np.asarray(h, dtype=np.float32)
    h0 = bf16_rne(h)
    r1 = (h - h0).astype(np.float32)
    h1 = bf16_rne(r1)
    r2 = (r1 - h1).astype(np.float32)
    h2 = bf16_rne(r2)
    return h0, h1, h2, r2


def test_three_bf16_terms_reconstruct_fp32_exactly():
    rng = np.random.default_rng(7)
    # magnitudes across the normal range, both signs, plus values that round up across a
    # power of two and the largest bf16 boundary cases
    mant = rng.random(200_000, dtype=np.float32) + 1.0
    expo = rng.integers(-100, 100, size=mant.size)
    h = (np.ldexp(mant, expo) * rng.choice([-1, 1], size=mant.size)).astype(np.float32)
    edge = np.array([1.0, -1.0, 1.0 + 2.0 ** -23, 2.0 - 2.0 ** -23, 1.0 + 2.0 ** -8,
                     1.0 + 2.0 ** -9, 1.0 + 2.0 ** -9 + 2.0 ** -23, 3.0e38, -2.5e-33],
                    dtype=np.float32)
    h = np.concatenate([h, edge])
    h0, h1, h2, r2 = split3(h)
    # the last remainder is already a bf16 value, so nothing is lost
    np.testing.assert_array_equal(h2, r2)
    total = h0.astype(np.float64) + h1.astype(np.float64) + h2.astype(np.float64)
    np.testing.assert_array_equal(total, h.astype(np.float64))
    # and each term is a bf16 value
    for t in (h0, h1, h2):
        assert np.all((t.view(np.uint32) & 0xFFFF) == 0)


def test_bf16_products_are_exact_in_fp32():
    rng = np.random.default_rng(8)
    a = bf16_rne(rng.normal(0, 3, 100_000).astype(np.float32))
    b = bf16_rne(rng.normal(0, 0.02, 100_000).astype(np.float32))
    prod32 = (a * b).astype(np.float32)
    np.testing.assert_array_equal(prod32.astype(np.float64), a.astype(np.float64) * b.astype(np.float64))
