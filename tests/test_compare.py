"""The comparison helpers themselves (CPU)."""
import numpy as np
import pytest

from tests.compare import bf16_order, check_bf16, check_f32


def test_bf16_order_across_zero():
    bits = np.array([0x8001, 0x8000, 0x0000, 0x0001, 0x3F80, 0x3F81], np.uint16)
    assert bf16_order(bits).tolist() == [-1, 0, 0, 1, 0x3F80, 0x3F81]


def test_check_bf16_limits():
    a = np.arange(0x3F00, 0x3F00 + 20000, dtype=np.uint16)
    check_bf16(a.copy(), a)
    b = a.copy()
    b[0] += 1
    check_bf16(b, a)                 # 1 of 20000 differs by 1 ulp: 99.995% identical
    b[1] += 2
    with pytest.raises(AssertionError):
        check_bf16(b, a)
    c = a.copy()
    c[:3] += 1                       # 99.985% identical
    with pytest.raises(AssertionError):
        check_bf16(c, a)


def test_check_f32():
    w = np.array([1.0, -2.0], np.float32)
    check_f32(w + np.float32(1e-6), w, 1.0, 1)
    with pytest.raises(AssertionError):
        check_f32(w + np.float32(1e-5), w, 1.0, 1)


def test_tally_judges_the_total():
    from tests.compare import Bf16Tally
    t = Bf16Tally()
    a = np.arange(0x3F00, 0x3F00 + 7, dtype=np.uint16)
    b = a.copy()
    b[0] += 1
    t.add(b, a)                      # one tiny key: 6 of 7 identical
    big = np.arange(0, 60000, dtype=np.uint16)
    t.add(big.copy(), big)
    assert t.frac() > 0.9999
    t.check()


def test_f32_to_bf16_bound():
    from tests.compare import check_f32_to_bf16
    a = np.array([0x3F80, 0x0001, 0xBC00], np.uint16)
    b = a.copy()
    b[0] += 1                         # one ulp at 1.0: inside
    assert check_f32_to_bf16(b, a, 0.05, 4) == 1
    c = a.copy()
    c[0] += 3                         # three ulps at 1.0 (0.023) > 2e-7 + 0.0078
    with pytest.raises(AssertionError):
        check_f32_to_bf16(c, a, 0.05, 4)
