"""The pre-pass computes the block scale s = RN(amax / 448) without a
division: q0 = RN(amax * y), r = RN(amax - 448 * q0) (exact in a fused
multiply-add), s = RN(q0 + r * y) with y = RN(1 / 448) (Markstein, IBM J.
Res. Dev. 34(1), 1990).  Checked here in exact rational arithmetic against
the correctly rounded float32 quotient over seeded maxima across the range the
kernel uses it for (2^-90 .. 2^100) and at the boundaries of every binade."""
from fractions import Fraction as F
import random

import numpy as np


def rn32(x: F) -> F:
    """Round a rational to the nearest float32 (ties to even), normal range."""
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if F(2) ** e > x:
        e -= 1
    while F(2) ** (e + 1) <= x:
        e += 1
    ulp = F(2) ** (e - 23)
    m = x / ulp
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > F(1, 2) or (rem == F(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def corrected_quotient(a: F, b: F, y: F) -> F:
    q0 = rn32(a * y)
    r = rn32(a - q0 * b)
    return rn32(q0 + r * y)


def test_rn32_matches_numpy():
    rng = np.random.default_rng(0)
    for v in rng.standard_normal(200) * 10.0 ** rng.integers(-20, 20, 200):
        assert float(rn32(F(float(v)))) == float(np.float32(v))


def test_scale_by_corrected_quotient_is_correctly_rounded():
    y = rn32(F(1, 448))
    assert float(y) == float(np.float32(1) / np.float32(448))
    random.seed(1)
    vals = [F(float(np.float32(random.uniform(1, 2) * 2.0 ** random.randint(-90, 99)))) for _ in range(3000)]
    for k in range(-90, 100, 7):
        vals.append(F(2) ** k)
        vals.append(F(float(np.nextafter(np.float32(2.0 ** k), np.float32(0)))))
        vals.append(F(float(np.nextafter(np.float32(448.0 * 2.0 ** (k - 9)), np.float32(np.inf)))))
    for a in vals:
        assert corrected_quotient(a, F(448), y) == rn32(a / 448), float(a)
