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


def _bits(vals):
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_fp32_sum_model_hand_case():
    """3*1 + 5*2 = 13, / 8 = 1.625, exact in every format."""
    from tests.compare import fp32_sum_model
    xs = [_bits([1.0]), _bits([2.0])]
    assert fp32_sum_model([3.0, 5.0], [True, True], xs, "f32")[0] == np.float32(1.625)
    assert fp32_sum_model([3.0, 5.0], [True, True], xs, "bf16")[0] == _bits([1.625])[0]
    # a client that did not report contributes nothing, and is not in N
    xs3 = xs + [_bits([100.0])]
    assert fp32_sum_model([3.0, 5.0, 7.0], [True, True, False], xs3, "f32")[0] == np.float32(1.625)


def test_fp32_sum_model_keeps_sequential_rounding():
    """2^24 + 1 rounds back to 2^24 in fp32 (ties to even), so 2^24 + 1 - 2^24 is 0 in
    the fp32 sum while the exact mean is 1/3: the model must show the fp32 result."""
    from tests.compare import fp32_sum_model
    xs = [_bits([2.0 ** 24]), _bits([1.0]), _bits([-(2.0 ** 24)])]
    assert fp32_sum_model([1.0, 1.0, 1.0], [True] * 3, xs, "f32")[0] == 0.0
    import oracle
    y, _, _ = oracle.fedavg_key([1.0, 1.0, 1.0], [True] * 3, xs, "bf16", "f32")
    assert y[0] == np.float32(1.0 / 3.0)


def test_tally_accepts_beyond_one_ulp_only_where_the_fp32_sum_explains_it():
    from tests.compare import Bf16Tally
    want = np.array([0x3F80, 0x3F80], np.uint16)
    got = want.copy()
    got[1] += 10                                  # 10 ulps at 1.0 (0.078)
    model = got.copy()
    t = Bf16Tally()
    t.add(got, want, "explained", model=model, bound=0.1)
    assert t.beyond == 1
    with pytest.raises(AssertionError):           # no model: the plain rule
        Bf16Tally().add(got, want, "plain")
    with pytest.raises(AssertionError):           # the model disagrees with the device
        Bf16Tally().add(got, want, "unexplained", model=want, bound=0.1)
    with pytest.raises(AssertionError):           # beyond the fp32 bound
        Bf16Tally().add(got, want, "too far", model=model, bound=1e-3)
