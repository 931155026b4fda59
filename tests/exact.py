"""Exact (rational) reference helpers for pinning the oracle.

Independent of the oracle's code: values are Fractions, and rounding picks the
nearest representable value by binary search over the target format's bit
patterns, decoded exactly.  Slow; for small cases only."""
from fractions import Fraction
import math
import struct


def f32_bits_to_fraction(b: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", b))[0])


def bf16_bits_to_fraction(b: int) -> Fraction:
    return f32_bits_to_fraction((b & 0xFFFF) << 16)


def _nearest_bits(v: Fraction, decode, max_finite_bits: int, inf_bits: int, sign_bit: int) -> int:
    """Nearest value of a binary floating-point format to v, ties to even bits."""
    neg = v < 0
    a = -v if neg else v
    sign = sign_bit if neg else 0
    lo, hi = 0, max_finite_bits           # largest pattern with value <= a
    if a >= decode(max_finite_bits):
        lo = max_finite_bits
    else:
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if decode(mid) <= a:
                lo = mid
            else:
                hi = mid
        if decode(hi) <= a:
            lo = hi
    below = decode(lo)
    if below == a:
        return sign | lo
    if lo == max_finite_bits:
        # next value above the largest finite is "one quantum higher", i.e. 2^(emax+1)
        q = decode(max_finite_bits) - decode(max_finite_bits - 1)
        above = below + q
        up_bits = inf_bits
    else:
        above = decode(lo + 1)
        up_bits = lo + 1
    d_lo, d_hi = a - below, above - a
    if d_lo < d_hi:
        return sign | lo
    if d_hi < d_lo:
        return sign | up_bits
    return sign | (lo if lo % 2 == 0 else up_bits)


def nearest_bf16(v: Fraction) -> int:
    return _nearest_bits(v, bf16_bits_to_fraction, 0x7F7F, 0x7F80, 0x8000)


def nearest_f32(v: Fraction) -> int:
    return _nearest_bits(v, f32_bits_to_fraction, 0x7F7FFFFF, 0x7F800000, 0x80000000)


def f32_to_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def exact_fedavg(weights, reported, values):
    """values[k] = list of Fractions (or floats) for one key; returns list of Fractions or None."""
    N = sum(Fraction(weights[k]) for k in range(len(weights)) if reported[k])
    if N == 0:
        return None
    m = len(next(v for k, v in enumerate(values) if reported[k]))
    out = []
    for i in range(m):
        s = sum(Fraction(weights[k]) * Fraction(values[k][i])
                for k in range(len(weights)) if reported[k])
        out.append(s / N)
    return out
