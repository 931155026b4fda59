"""Hierarchical FedAvg (silos, then a mean over silos weighted by each silo's total):
the summary "Adaptive Data Partitioning for Energy-Efficient Federated and
Distributed Learning in Heterogeneous Systems", section 2, "Execution regimes",
item 3 (HFL-DDP): silo models are aggregated at federated round boundaries.
In exact arithmetic the two-level mean equals the flat weighted mean over all
clients; the oracle's fp64 nesting must agree with its flat form to fp64
rounding, and both must round to the same outputs."""
from fractions import Fraction

import numpy as np

import oracle
from tests import exact


def test_two_level_equals_flat():
    rng = np.random.default_rng(41)
    K, m = 11, 4000
    w = [float(v) for v in rng.integers(50, 5000, K)]
    xs = [((rng.standard_normal(m) * 0.02).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
          for _ in range(K)]
    silos = [[0, 1, 2], [3, 4, 5, 6], [7], [8, 9, 10]]
    nested = oracle.hierarchical_f64(silos, w, [True] * K, xs, "bf16")
    flat = oracle.fedavg_key_f64(w, [True] * K, xs, "bf16")
    # fp64 rounding of a few operations, scaled to the inputs (results near zero cancel)
    scale = max(float(np.abs((x.astype(np.uint32) << 16).view(np.float32)).max()) for x in xs)
    assert np.max(np.abs(nested - flat)) <= 64 * 2.0 ** -52 * scale
    a = oracle.bf16_rne(nested)
    b = oracle.bf16_rne(flat)
    assert np.mean(a == b) >= 0.9999


def test_two_level_exact_small():
    """Exact rationals: the mean of silo means weighted by silo totals is the flat mean."""
    rng = np.random.default_rng(42)
    for _ in range(20):
        K = int(rng.integers(2, 7))
        w = [int(v) for v in rng.integers(1, 100, K)]
        x = [[Fraction(int(v), 64) for v in rng.integers(-64, 64, 3)] for _ in range(K)]
        cut = int(rng.integers(1, K))
        silos = [list(range(cut)), list(range(cut, K))]
        flat = exact.exact_fedavg(w, [True] * K, x)
        means = [exact.exact_fedavg([w[k] for k in s], [True] * len(s), [x[k] for k in s]) for s in silos]
        tot = [sum(w[k] for k in s) for s in silos]
        assert exact.exact_fedavg(tot, [True, True], means) == flat
        # and the fp64 oracle nesting rounds to the exact value's nearest binary32
        xs = [np.array([float(v) for v in xi], np.float32) for xi in x]
        nested = oracle.hierarchical_f64(silos, [float(v) for v in w], [True] * K, xs, "f32")
        assert oracle.f32_rn(nested).view(np.uint32).tolist() == [exact.nearest_f32(v) for v in flat]


def test_silo_without_weight_is_skipped():
    xs = [np.array([1.0, 2.0], np.float32), np.array([5.0, 5.0], np.float32), np.array([3.0, 4.0], np.float32)]
    nested = oracle.hierarchical_f64([[0], [1], [2]], [2.0, 0.0, 2.0], [True] * 3, xs, "f32")
    assert nested.tolist() == [2.0, 3.0]
