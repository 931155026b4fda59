"""Tolerances the GPU path is held to against the fp64 oracle.

  fp32 output: |gpu - oracle| <= 1e-6 * max|w| * K per element, where max|w| is
               the largest input magnitude over the key's reporters and K the
               number of clients that reported the key;
  bf16 output: at most 1 bf16 ulp apart everywhere, and >= 99.99% of elements
               bit-identical (+0 and -0 count as equal);
  totals / masks: bit-exact.
"""
import numpy as np

BF16_MIN_IDENTICAL = 0.9999


def bf16_order(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that are consecutive for adjacent values
    (so |a - b| counts ulps across zero); -0 and +0 both map to 0."""
    b = bits.astype(np.int64) & 0xFFFF
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


class Bf16Tally:
    """Accumulates bf16 comparisons over a whole workload: every element within
    1 ulp (checked per call), the identical fraction checked over the total."""

    def __init__(self):
        self.same = 0
        self.total = 0

    def add(self, got_bits: np.ndarray, want_bits: np.ndarray, what: str = ""):
        g = bf16_order(got_bits.view(np.uint16) if got_bits.dtype != np.uint16 else got_bits)
        w = bf16_order(want_bits)
        d = np.abs(g - w)
        assert d.size == 0 or int(d.max()) <= 1, f"{what}: bf16 differs by {int(d.max())} ulp"
        self.same += int(np.count_nonzero(d == 0))
        self.total += int(d.size)

    def frac(self) -> float:
        return 1.0 if self.total == 0 else self.same / self.total

    def check(self, what: str = "", minimum: float = BF16_MIN_IDENTICAL) -> float:
        f = self.frac()
        assert f >= minimum, f"{what}: only {f:.6%} of {self.total} bf16 elements bit-identical"
        return f


def check_bf16(got_bits: np.ndarray, want_bits: np.ndarray, what: str = "") -> float:
    t = Bf16Tally()
    t.add(got_bits, want_bits, what)
    return t.check(what)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_f32_to_bf16(got_bits, want_bits, max_abs_in: float, K: int, what: str = "") -> int:
    """fp32 inputs, bf16 output: the fp32 running-sum bound plus one bf16 ulp of the
    result.  (With fp32 inputs the products n_k*x round inside the sum, so near-total
    cancellation can move a small result by several bf16 ulps; the bf16 rule above
    is for bf16 inputs, whose products are exact.)  Returns the number of elements
    that are not bit-identical."""
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
