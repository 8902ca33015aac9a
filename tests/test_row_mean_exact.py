"""The LayerNorm kernels form a row's mean as q = RN(total * y) with
y = RN(1 / n), refined once: q' = RN(q + RN(total - q * n) * y), where the
remainder total - q * n is exact in one fma.  A constant row relies on this
returning a quotient that is a float exactly (its sum n * c is exact, so
x - mu must come out 0 and the output must be the shift bit for bit).

This checks that arithmetic on the CPU, each f32 rounding done exactly with
rationals, for every 7th bf16 value c in [2^-10, 2^10) at the row widths the
tests and benchmarks use, and that the remainder is always exact.  No GPU."""
from fractions import Fraction

import numpy as np
import pytest


def rn_f32(x):
    """Round a rational to the nearest f32, ties to even (normal range)."""
    d = np.float32(float(x))  # float() rounds once to double, then to f32
    best = None
    for c in (np.nextafter(d, np.float32(-np.inf)), d, np.nextafter(d, np.float32(np.inf))):
        err = abs(Fraction(float(c)) - x)
        odd = int(np.float32(c).view(np.uint32)) & 1
        key = (err, odd)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def refined_mean(total, n):
    y = rn_f32(Fraction(1, n))
    q = rn_f32(Fraction(float(total)) * Fraction(float(y)))
    exact_r = Fraction(float(total)) - Fraction(float(q)) * n
    r = rn_f32(exact_r)
    assert Fraction(float(r)) == exact_r, "the remainder must be exact"
    return rn_f32(Fraction(float(q)) + Fraction(float(r)) * Fraction(float(y)))


BF16_VALUES = (np.arange(0x3A80, 0x4480, 7, dtype=np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("n", [8, 24, 64, 1000, 1024, 3000, 3072, 4096, 5120, 8192, 12288, 32768])
def test_constant_row_mean_is_exact(n):
    checked = 0
    for c in BF16_VALUES:
        total = Fraction(float(c)) * n
        if Fraction(float(rn_f32(total))) != total:
            continue  # n * c not a float: the sum itself would round
        assert refined_mean(np.float32(float(total)), n) == c, (float(c), n)
        checked += 1
    assert checked > 100


def test_a_plain_product_is_not_always_exact():
    """Without the refinement step the product RN(total * y) misses: the
    step is what makes the claim hold (so the test above can fail)."""
    misses = 0
    for n in (1000, 3000, 3072, 5120, 12288):
        y = rn_f32(Fraction(1, n))
        for c in BF16_VALUES:
            total = Fraction(float(c)) * n
            if Fraction(float(rn_f32(total))) != total:
                continue
            if rn_f32(total * Fraction(float(y))) != c:
                misses += 1
    assert misses > 0
