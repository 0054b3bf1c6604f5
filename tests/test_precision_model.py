"""Host model of the band path's split-operand arithmetic.

The window's product A Z_k runs on bf16 tensor cores with each operand split
into two bf16 parts, x = hi + lo with hi = RN_bf16(x) and lo = RN_bf16(x - hi),
and three of the four partial products (e_hi z_hi + e_hi z_lo + e_lo z_hi,
fp32 accumulation).  The precision argument for the 4e-3 output budget rests
on this carrying each weight-value product to about 2^-16 relative; here the
same roundings are applied in numpy and the claim is checked against fp64.
"""
import numpy as np

from sparse_long_sequence_gb300 import synthetic


def bf16(x):
    """Round to nearest-even bfloat16 (through float32, as the kernels do)."""
    return synthetic.bf16_bits_to_f32(synthetic.to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def split(x):
    hi = bf16(x)
    lo = bf16(np.asarray(x, np.float32).astype(np.float64) - hi)
    return hi, lo


def test_two_part_split_carries_sixteen_bits():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200_000).astype(np.float32).astype(np.float64)
    hi, lo = split(x)
    rel = np.abs(x - hi - lo) / np.abs(x)
    assert rel.max() <= 2.0 ** -16
    assert np.abs(x - hi).max() / np.abs(x).max() > 2.0 ** -10     # one part alone is not enough


def test_three_product_dot_within_budget():
    # a window row: 513 weights e in (0, 1] against Z_k rows of unit scale; the
    # split product sum against the exact fp64 sum, relative to sum_j e_j |z_j|
    rng = np.random.default_rng(1)
    for _ in range(50):
        e = np.exp(-rng.exponential(2.0, 513)).astype(np.float32).astype(np.float64)
        z = rng.standard_normal(513).astype(np.float32).astype(np.float64)
        eh, el = split(e)
        zh, zl = split(z)
        approx = np.sum((eh * zh).astype(np.float32)) + np.sum((eh * zl).astype(np.float32)) + \
            np.sum((el * zh).astype(np.float32))
        exact = np.sum(e * z)
        assert abs(approx - exact) <= 2.0 ** -14 * np.sum(e * np.abs(z))


def test_output_rounding_uses_most_of_the_budget():
    # RN to bf16 alone: up to 2^-8 of |x| (half an ulp at 8 significant bits, for
    # x just above a power of two), 3.9e-3 of the 4e-3 row budget: the arithmetic
    # before it must stay near 1e-4
    rng = np.random.default_rng(2)
    x = rng.standard_normal(200_000).astype(np.float32).astype(np.float64)
    rel = np.abs(bf16(x) - x) / np.abs(x)
    assert rel.max() <= 2.0 ** -8 and rel.max() > 2.0 ** -8 * 0.99
