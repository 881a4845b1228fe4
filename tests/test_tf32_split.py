"""The error bound of the three-way tf32 split that the fp32 tensor-core decode
step relies on, checked from the definitions on the host.

tf32 keeps the sign, the 8-bit exponent and the top 10 bits of an fp32
significand. hi = x rounded to the nearest tf32 (ties away from zero, as
cvt.rna), lo = x - hi (exact in fp32), and the tensor core reads lo with its
low 13 significand bits dropped. A product a b is taken as
ah bh + ah bl + al bh. The claim: the result is within 2^-19 of |a b| (the
dropped al bl is below 2^-22 of it, lo's truncation below 2^-21 in each of the
two cross terms), far inside the 1e-5 bound of the fp32 path.
"""
import numpy as np

MASK_TF32 = np.uint32(0xFFFFE000)


def to_tf32_rna(x):
    """Round fp32 values to the nearest tf32, ties away from zero."""
    b = x.astype(np.float32).view(np.uint32)
    # add half of the dropped range to the magnitude bits, then truncate (sign bit untouched)
    r = (b & np.uint32(0x7FFFFFFF)) + np.uint32(0x1000)
    return ((r & MASK_TF32) | (b & np.uint32(0x80000000))).view(np.float32)


def truncate_tf32(x):
    return (x.astype(np.float32).view(np.uint32) & MASK_TF32).view(np.float32)


def split(x):
    hi = to_tf32_rna(x)
    lo = (x.astype(np.float32) - hi).astype(np.float32)
    return hi, lo


def test_hi_is_a_tf32_value_and_lo_is_exact():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * np.exp2(rng.integers(-20, 20, 100000))).astype(np.float32)
    hi, lo = split(x)
    assert np.all((hi.view(np.uint32) & np.uint32(0x1FFF)) == 0)
    # x = hi + lo exactly: the difference of x and its rounding has at most 13 significant bits
    assert np.array_equal((hi.astype(np.float64) + lo.astype(np.float64)).astype(np.float32), x)
    assert np.all(np.abs(lo) <= np.abs(x) * 2.0 ** -11)


def test_three_products_are_within_the_bound():
    rng = np.random.default_rng(1)
    a = (rng.standard_normal(200000) * np.exp2(rng.integers(-8, 8, 200000))).astype(np.float32)
    b = (rng.standard_normal(200000) * np.exp2(rng.integers(-8, 8, 200000))).astype(np.float32)
    ah, al = split(a)
    bh, bl = split(b)
    al_t, bl_t = truncate_tf32(al).astype(np.float64), truncate_tf32(bl).astype(np.float64)
    approx = ah.astype(np.float64) * bh + ah.astype(np.float64) * bl_t + al_t * bh.astype(np.float64)
    exact = a.astype(np.float64) * b.astype(np.float64)
    err = np.abs(approx - exact)
    assert np.all(err <= np.abs(exact) * 2.0 ** -19)
    # one product of tf32 values alone would not do: its error reaches past 2^-13 of |a b|
    one = np.abs(ah.astype(np.float64) * bh - exact)
    assert np.any(one > np.abs(exact) * 2.0 ** -13)
