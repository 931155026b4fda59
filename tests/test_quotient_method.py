"""The division-free quotient of the final form, checked as arithmetic on the CPU: Markstein's
correction of a reciprocal (P. Markstein, IBM J. Res. Develop. 34(1), 1990), taken twice,
in exact rational arithmetic with every fp32 rounding done explicitly, against the exactly
rounded quotient RN(s/d).  The GPU suite checks the kernel itself on every fp32 sum for a
few divisors; this checks the method over random and adversarial (near-midpoint) operands
across the whole range the kernel admits (2^-60 <= |s| < 2^61, 2^-20 <= d <= 2^60)."""
import random
from fractions import Fraction

import pytest

P = 24      # fp32 significand bits


def rn32(x: Fraction) -> Fraction:
    """x rounded to the nearest fp32 value, ties to even (normal range only)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert -126 <= e <= 127, "outside the normal range"
    scale = Fraction(2) ** (e - (P - 1))      # one ulp at this binade
    m = a / scale                             # in [2^23, 2^24)
    q, r = divmod(m.numerator, m.denominator)
    rem = Fraction(r, m.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and q % 2 == 1):
        q += 1
    return sign * q * scale


def fma32(a, b, c):
    return rn32(a * b + c)


def markstein(s: Fraction, d: Fraction) -> Fraction:
    y = rn32(1 / d)
    q = rn32(s * y)
    q = fma32(fma32(-q, d, s), y, q)
    return fma32(fma32(-q, d, s), y, q)


def rand_f32(rng, lo_exp, hi_exp, integer=False):
    if integer:
        return Fraction(rng.randint(1, (1 << 24) - 1))
    m = rng.randint(1 << 23, (1 << 24) - 1)
    e = rng.randint(lo_exp, hi_exp)
    return m * Fraction(2) ** (e - 23)


def test_rn32_rounds_to_nearest_even():
    one = Fraction(1)
    ulp = Fraction(2) ** -23
    assert rn32(one + ulp / 2) == one                 # tie: to even
    assert rn32(one + 3 * ulp / 2) == one + 2 * ulp   # tie: to even (up)
    assert rn32(one + ulp / 2 + ulp / 1024) == one + ulp
    assert rn32(Fraction(1, 3)) == Fraction(11184811, 33554432)   # 0x3EAAAAAB


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_operands(seed):
    rng = random.Random(seed)
    for _ in range(3000):
        d = rand_f32(rng, -20, 59, integer=rng.random() < 0.4)
        s = rand_f32(rng, -60, 60) * (1 if rng.random() < 0.5 else -1)
        assert markstein(s, d) == rn32(s / d), (s, d)


def test_quotients_next_to_rounding_midpoints():
    """The hardest operands: s/d as close to a midpoint between two floats as a quotient of
    two floats can be, 1/(2D) ulps for a divisor with odd significand D.  With D odd and
    M = 2^24 + (-+D^-1 mod 2^24) (odd), S = (M*D +- 1) / 2^24 is an integer; for
    2^23 <= S < 2^24, s = S*2^23 and d = D give s/d = M/2 +- 1/(2D), M/2 a midpoint of floats
    in [2^23, 2^24).  Scaled by powers of two across the admitted range.  The product by the
    reciprocal alone rounds many of these the wrong way; the two corrections get every one
    right."""
    rng = random.Random(7)
    n = wrong_product = 0
    while n < 600:
        D = rng.randrange((1 << 22) + 1, 1 << 24, 2)
        inv = pow(D, -1, 1 << 24)
        sign = rng.choice((1, -1))
        M = (1 << 24) + ((-sign * inv) % (1 << 24))
        num = M * D + sign
        assert num % (1 << 24) == 0 and M % 2 == 1
        S = num >> 24
        if not (1 << 23) <= S < (1 << 24):
            continue
        ds = rng.randint(-20, 36)                    # d = D * 2^ds within [2^-20, 2^60]
        ss = rng.randint(-60 - 23 + ds + 24, 36)    # keeps 2^-60 <= |s| < 2^61
        d = D * Fraction(2) ** (ds - 23)
        s = S * Fraction(2) ** (ss) * (1 if rng.random() < 0.5 else -1)
        if not (Fraction(2) ** -60 <= abs(s) < Fraction(2) ** 61 and Fraction(2) ** -20 <= d <= Fraction(2) ** 60):
            continue
        want = rn32(s / d)
        assert markstein(s, d) == want, (s, d)
        wrong_product += rn32(s * rn32(1 / d)) != want
        n += 1
    assert wrong_product > n // 10
