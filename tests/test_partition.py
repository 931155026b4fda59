"""Adaptive allocation controller (the library's fa_partition_plan, host code) against
its plain oracle, hand-worked allocations, and the properties the page states:
samples go inversely proportional to cost, the budget is fixed, every participant
is kept, a deadband suppresses negligible reallocation."""
import math
import random

import pytest

import server_side_fedavg_gb300 as fa
from oracle.partition import partition_plan


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import os
    if not os.path.exists(fa.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()


def test_hand_worked_time_only():
    # tau = (1, 2, 4) s/sample, median 2 -> c = (0.5, 1, 2) -> shares (4/7, 2/7, 1/7);
    # 30 samples: one each, then 27 * shares = (15.43, 7.71, 3.86) -> floors (15, 7, 3),
    # two left by largest fraction (0.86, 0.71) -> (15, 8, 4) -> +1 each -> (16, 9, 5)
    want = [16, 9, 5]
    assert partition_plan([10.0, 20.0, 40.0], [0.0] * 3, [10, 10, 10])[0] == want
    got, tau, eps = fa.fa_partition_plan([10.0, 20.0, 40.0], [0.0] * 3, [10, 10, 10])
    assert got == want and tau == [1.0, 2.0, 4.0]


def test_hand_worked_energy_and_ema():
    # round 1: equal time, energy per sample (1, 3): w_e = 1 only -> c = (0.5, 1.5) ->
    # shares (0.75, 0.25) of 20 -> 1 + 18*(0.75, 0.25) = (14.5 -> 14, 5.5 -> 5), one left,
    # equal fractions -> lower index -> (15, 5)
    n1, tau, eps = partition_plan([5.0, 5.0], [10.0, 30.0], [10, 10], w_time=0.0, w_energy=1.0)
    assert n1 == [15, 5] and eps == [1.0, 3.0]
    # round 2 (alpha 0.5): new eps (15/15, 15/5) = (1, 3) -> ema stays (1, 3); shares already
    # (0.75, 0.25) -> inside the deadband -> unchanged
    n2, tau2, eps2 = partition_plan([7.5, 2.5], [15.0, 15.0], n1, tau, eps, w_time=0.0, w_energy=1.0)
    assert n2 == [15, 5] and eps2 == [1.0, 3.0]


def test_hand_worked_zero_median_falls_back_to_the_mean():
    # time and energy weighted equally (w_t = w_e = 1), 10 samples each.
    # tau = t / n = (0, 0, 6): median 0 -> mean 2 -> normalised (0, 0, 3)
    # eps = e / n = (1, 2, 4): median 2 -> normalised (0.5, 1, 2)
    # c = (0.5, 1, 5) -> 1/c = (2, 1, 0.2), sum 3.2 -> shares (0.625, 0.3125, 0.0625)
    # 27 left after one each: (16.875, 8.4375, 1.6875) -> floors (16, 8, 1), two left by
    # largest fraction (0.875, 0.6875) -> (17, 8, 2) -> +1 each -> (18, 9, 3)
    args = ([0.0, 0.0, 60.0], [10.0, 20.0, 40.0], [10, 10, 10])
    kw = dict(w_time=1.0, w_energy=1.0)
    want = [18, 9, 3]
    assert partition_plan(*args, **kw)[0] == want
    assert fa.fa_partition_plan(*args, **kw)[0] == want


def test_hand_worked_all_zero_column_counts_as_ones():
    # no energy reported (all zero, median and mean 0): that column normalises to
    # (1, 1, 1) and no longer discriminates.  tau = (0, 2, 2): median 2 -> (0, 1, 1).
    # w_t = w_e = 0.5: c = (0.5, 1, 1) -> 1/c = (2, 1, 1), shares (0.5, 0.25, 0.25)
    # 27 left: (13.5, 6.75, 6.75) -> floors (13, 6, 6), two left by largest fraction
    # (0.75, 0.75 at the lower indices 1, 2) -> (13, 7, 7) -> +1 each -> (14, 8, 8)
    args = ([0.0, 20.0, 20.0], [0.0, 0.0, 0.0], [10, 10, 10])
    kw = dict(w_time=0.5, w_energy=0.5)
    want = [14, 8, 8]
    assert partition_plan(*args, **kw)[0] == want
    assert fa.fa_partition_plan(*args, **kw)[0] == want


def test_deadband_keeps_allocation():
    n, _, _ = partition_plan([10.0, 10.5, 9.8], [0.0] * 3, [100, 100, 100])
    assert n == [100, 100, 100]
    got, _, _ = fa.fa_partition_plan([10.0, 10.5, 9.8], [0.0] * 3, [100, 100, 100])
    assert got == [100, 100, 100]


@pytest.mark.parametrize("seed", range(20))
def test_library_matches_oracle(seed):
    rng = random.Random(seed)
    m = rng.randint(1, 11)
    samples = [rng.randint(1, 2000) for _ in range(m)]
    t = [rng.uniform(0.1, 100.0) * s for s in samples]
    e = [rng.uniform(0.0, 50.0) * s for s in samples]
    wt, we = rng.choice([(1.0, 0.0), (0.0, 1.0), (1.0, 0.25), (0.5, 0.5)])
    alpha, band = rng.choice([0.5, 0.3, 1.0]), rng.choice([0.0, 0.05, 0.2])
    tau = eps = None
    for rnd in range(3):
        want = partition_plan(t, e, samples, tau, eps, wt, we, alpha, band)
        got = fa.fa_partition_plan(t, e, samples, tau, eps, wt, we, alpha, band)
        assert got[0] == want[0]
        assert all(math.isclose(a, b, rel_tol=1e-14) for a, b in zip(got[1], want[1]))
        assert all(math.isclose(a, b, rel_tol=1e-14, abs_tol=1e-300) for a, b in zip(got[2], want[2]))
        samples, tau, eps = want
        t = [rng.uniform(0.1, 100.0) * s for s in samples]
        e = [rng.uniform(0.0, 50.0) * s for s in samples]


def test_properties():
    rng = random.Random(3)
    for _ in range(200):
        m = rng.randint(2, 12)
        samples = [rng.randint(1, 500) for _ in range(m)]
        t = [rng.uniform(0.01, 10.0) * s for s in samples]
        new, tau, _ = partition_plan(t, [0.0] * m, samples, deadband=0.0)
        assert sum(new) == sum(samples) and min(new) >= 1
        # inverse proportionality: a strictly cheaper participant never gets fewer samples
        for i in range(m):
            for j in range(m):
                if tau[i] < tau[j]:
                    assert new[i] >= new[j]


def test_invalid_arguments():
    with pytest.raises(fa.FedAvgError):
        fa.fa_partition_plan([1.0], [1.0], [0])
    with pytest.raises(fa.FedAvgError):
        fa.fa_partition_plan([-1.0], [1.0], [5])
    with pytest.raises(fa.FedAvgError):
        fa.fa_partition_plan([1.0], [1.0], [5], w_time=0.0, w_energy=0.0)
    with pytest.raises(fa.FedAvgError):
        fa.fa_partition_plan([1.0], [1.0], [5], ema_alpha=0.0)
