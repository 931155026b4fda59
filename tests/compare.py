"""Tolerances the GPU path is held to against the fp64 oracle.

  fp32 output: |gpu - oracle| <= 1e-6 * max|w| * K per element, where max|w| is
               the largest input magnitude over the key's reporters and K the
               number of clients that reported the key;
  bf16 output: at most 1 bf16 ulp apart, and >= 99.99% of elements
               bit-identical (+0 and -0 count as equal).  The one exception is the
               fp32 running sum's own rounding: where sum_k n_k*x_k nearly cancels
               (terms 1e6 times the result), the fp32 sum the method fixes can be
               many bf16 ulps from the exact mean.  An element may then be more than
               1 ulp away only if it equals, bit for bit, fp32_sum_model -- an
               independent model of that fp32 arithmetic -- and stays within the
               fp32 bound 1e-6 * max|x| * K plus one bf16 ulp;
  totals / masks: bit-exact.
"""
import numpy as np

import oracle

BF16_MIN_IDENTICAL = 0.9999


def bf16_order(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that are consecutive for adjacent values
    (so |a - b| counts ulps across zero); -0 and +0 both map to 0."""
    b = bits.astype(np.int64) & 0xFFFF
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def fp32_sum_model(weights, reported, xs, dtype_out):
    """The fp32 arithmetic of the aggregation, element by element, for bf16 inputs (uint16
    bits) and weights whose products with them are exact in fp32: the first reporter's
    product, each later reporter's product added with one fp32 rounding (a fused
    multiply-add whose product is exact), in client-id order; then an IEEE fp32 division
    by (float)N and the output cast (RNE).  Used only to tell the fp32 sum's own rounding
    from a wrong result where the weighted sum nearly cancels."""
    acc = None
    N = 0.0
    for k, (n, rep) in enumerate(zip(weights, reported)):
        if not rep:
            continue
        N += n
        x = (np.asarray(xs[k]).astype(np.uint32) << 16).view(np.float32)
        p64 = np.float64(n) * x.astype(np.float64)
        p = p64.astype(np.float32)
        assert np.array_equal(p.astype(np.float64), p64, equal_nan=True), "product not exact in fp32"
        acc = p if acc is None else (acc + p).astype(np.float32)
    q = (acc / np.float32(N)).astype(np.float32)
    return q if dtype_out == "f32" else oracle.bf16_rne(q.astype(np.float64))


class Bf16Tally:
    """Accumulates bf16 comparisons over a whole workload: every element within
    1 ulp (checked per call) -- or, given `model` and `bound`, beyond it only where the
    fp32 sum's own rounding explains it (see the module docstring) -- and the
    identical fraction checked over the total."""

    def __init__(self):
        self.same = 0
        self.total = 0
        self.beyond = 0

    def add(self, got_bits: np.ndarray, want_bits: np.ndarray, what: str = "", model=None,
            bound=None):
        got_bits = got_bits.view(np.uint16) if got_bits.dtype != np.uint16 else got_bits
        g = bf16_order(got_bits)
        w = bf16_order(want_bits)
        d = np.abs(g - w)
        over = d > 1
        if over.any():
            assert model is not None and bound is not None, \
                f"{what}: bf16 differs by {int(d.max())} ulp"
            assert np.array_equal(got_bits[over], np.asarray(model)[over]), \
                f"{what}: {int(over.sum())} elements beyond 1 ulp that the fp32 sum does not explain"
            gv, wv = bf16_values(got_bits[over]), bf16_values(want_bits[over])
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(wv), 2.0 ** -126))) - 7)
            assert (np.abs(gv - wv) <= bound + ulp).all(), f"{what}: beyond the fp32 bound"
            self.beyond += int(over.sum())
        self.same += int(np.count_nonzero(d == 0))
        self.total += int(d.size)

    def frac(self) -> float:
        return 1.0 if self.total == 0 else self.same / self.total

    def check(self, what: str = "", minimum: float = BF16_MIN_IDENTICAL) -> float:
        f = self.frac()
        assert f >= minimum, f"{what}: only {f:.6%} of {self.total} bf16 elements bit-identical"
        return f


def check_bf16(got_bits: np.ndarray, want_bits: np.ndarray, what: str = "", model=None,
               bound=None) -> float:
    t = Bf16Tally()
    t.add(got_bits, want_bits, what, model, bound)
    if t.beyond:
        print(f"{what}: {t.beyond} element(s) beyond 1 ulp, each equal to the fp32 sum model")
    return t.check(what)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_f32_to_bf16(got_bits, want_bits, max_abs_in: float, K: int, what: str = "") -> int:
    """bf16 output where the products n_k*x are not exact in fp32 -- fp32 inputs, or
    weights with more than 16 significant bits (totals above 2^24) or not integers: the
    fp32 running-sum bound plus one bf16 ulp of the result.  (Those products round inside
    the sum, so near-total cancellation can move a small result by several bf16 ulps; the
    bf16 rule above is for bf16 inputs and integer weights up to 2^16, whose products are
    exact.)  Returns the number of elements that are not bit-identical."""
    g = bf16_values(got_bits.view(np.uint16))
    w = bf16_values(want_bits)
    mag = np.maximum(np.abs(w), 2.0 ** -126)
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    tol = 1e-6 * max_abs_in * K + ulp
    d = np.abs(g - w)
    bad = d > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond fp32 bound + 1 bf16 ulp"
    return int(np.count_nonzero(g != w))


def check_f32(got: np.ndarray, want: np.ndarray, max_abs_in: float, K: int, what: str = "") -> float:
    tol = 1e-6 * max_abs_in * K
    d = np.abs(got.astype(np.float64) - want.astype(np.float64))
    worst = float(d.max()) if d.size else 0.0
    assert worst <= tol, f"{what}: fp32 error {worst:.3e} > tol {tol:.3e}"
    return worst


def check_f32_compensated(got: np.ndarray, want: np.ndarray, max_abs_in: float, what: str = "") -> float:
    """fp32 output of the compensated mode (FA_COMPENSATED): its Dot2 sum is as accurate as
    one held in about twice fp32's precision (error at most ~K^2 * 2^-48 of the sum of
    |terms|, itself at most max|x| times the divisor), and the corrected division adds
    under one ulp of the quotient.  So every element is within two fp32 ulps of the
    oracle's correctly rounded value, plus 2^-38 * max|x| where the weighted sum nearly
    cancels.  Returns the largest error in ulps of the oracle value."""
    g = got.astype(np.float64)
    w = want.astype(np.float64)
    mag = np.maximum(np.abs(w), np.float64(np.finfo(np.float32).tiny))
    ulp = np.exp2(np.floor(np.log2(mag)) - 23)
    d = np.abs(g - w)
    tol = 2.0 * ulp + 2.0 ** -38 * max_abs_in
    bad = d > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond the compensated bound " \
                          f"(worst {float((d / ulp).max()):.1f} ulp)"
    return float((d / ulp).max()) if d.size else 0.0
