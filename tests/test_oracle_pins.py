"""Pins for the fp64 oracle: every check compares it with something other than
itself -- hand sums, a hand-made RNE table, exact rational arithmetic, a library
routine (numpy.average / numpy.mean), and invariants of the weighted mean.

The aggregation being pinned (weighted mean per key over the clients that
reported the key, weights = sample counts, RNE output cast) follows
"Federated learning implemented by NVIDIA Clara" (opening section and
"Server-side workflow"), the adaptive-partitioning summary's controller
("Measurement": n_i sample counts), the FLARE multimodal blog's client update
contract ("Coordinating training across clients"), and the NVFP4 blog's
rounding item (weights use round-to-nearest-even)."""
import itertools
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32(vals):
    return np.asarray(vals, dtype=np.float32)


def _bf16_bits(vals):
    """Exactly representable bf16 values -> bits (test inputs only)."""
    a = np.asarray(vals, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly bf16"
    return (u >> 16).astype(np.uint16)


def _random_bf16(rng, n, scale=1.0):
    f = (rng.standard_normal(n) * scale).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _bf16_to_f64(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------- golden hand sums
def _read_hand_sums():
    cases = []
    with open(os.path.join(GOLDEN, "hand_sums.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w, xs, exp = [p.strip() for p in line.split("|")]
            weights = [float(t) for t in w.split()]
            clients = [[float(t) for t in c.split()] for c in xs.split(";")]
            if len(clients) == 1 and len(weights) == 1:
                pass
            expected = [float(t) for t in exp.split()]
            cases.append((weights, clients, expected))
    return cases


@pytest.mark.parametrize("case", _read_hand_sums())
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_hand_sums(case, dt):
    weights, clients, expected = case
    K = len(weights)
    if len(clients) != K:          # single-client line with several elements
        clients = [clients[0]]
    conv = _f32 if dt == "f32" else _bf16_bits
    xs = [conv(c) for c in clients]
    out, N, cnt = oracle.fedavg_key(weights, [True] * K, xs, dt, dt)
    got = out.astype(np.float64) if dt == "f32" else _bf16_to_f64(out)
    assert got.tolist() == expected
    assert N == sum(weights) and cnt == K


# ----------------------------------------------------------------- RNE table
def _read_rne():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            expr, bits, note = [p.strip() for p in line.split("|")]
            rows.append((expr, int(bits, 16), note))
    return rows


@pytest.mark.parametrize("row", _read_rne(), ids=lambda r: r[0])
def test_bf16_rne_table(row):
    expr, bits, _ = row
    y = eval(expr, {"float": float})
    assert oracle.lib().fo_bf16_rne(y) == bits


def test_bf16_rne_nan():
    assert oracle.lib().fo_bf16_rne(float("nan")) & 0x7FFF == 0x7FC0


def test_bf16_rne_bruteforce():
    """Random doubles over the whole bf16 range against exact nearest-by-search."""
    rng = random.Random(7)
    ys = []
    for _ in range(3000):
        e = rng.uniform(-140, 129)
        ys.append(rng.choice([-1, 1]) * rng.random() * 2.0 ** e)
    # exact ties and neighbours around random bf16 values
    for _ in range(1000):
        b = rng.randrange(1, 0x7F7F)
        lo = float(exact.bf16_bits_to_fraction(b))
        hi = float(exact.bf16_bits_to_fraction(b + 1))
        mid = (lo + hi) / 2            # exact in fp64
        ys += [mid, math.nextafter(mid, 0), math.nextafter(mid, math.inf)]
    got = oracle.bf16_rne(ys)
    want = [exact.nearest_bf16(Fraction(y)) for y in ys]
    assert got.tolist() == want


def test_f32_rn_bruteforce():
    rng = random.Random(8)
    ys = [rng.choice([-1, 1]) * rng.random() * 2.0 ** rng.uniform(-140, 127) for _ in range(2000)]
    got = oracle.f32_rn(ys).view(np.uint32)
    want = [exact.nearest_f32(Fraction(y)) for y in ys]
    assert got.tolist() == want


# ----------------------------------------------------------------- exact rational FedAvg
@pytest.mark.parametrize("dt_in,dt_out", [("f32", "f32"), ("bf16", "bf16"), ("f32", "bf16"), ("bf16", "f32")])
def test_exact_rational(dt_in, dt_out):
    """Oracle output == the exactly computed weighted mean, rounded to nearest."""
    rng = np.random.default_rng(11)
    for trial in range(40):
        K = int(rng.integers(1, 7))
        m = int(rng.integers(1, 20))
        weights = [float(v) for v in rng.integers(0, 5000, K)]
        if trial % 5 == 0:
            weights[0] = 0.0
        reported = [bool(v) for v in rng.integers(0, 2, K)]
        reported[int(rng.integers(0, K))] = True
        scale = 10.0 ** rng.uniform(-6, 2)
        if dt_in == "f32":
            xs = [(rng.standard_normal(m) * scale).astype(np.float32) for _ in range(K)]
            vals = [x.astype(np.float64).tolist() for x in xs]
        else:
            xs = [_random_bf16(rng, m, scale) for _ in range(K)]
            vals = [_bf16_to_f64(x).tolist() for x in xs]
        out, N, cnt = oracle.fedavg_key(weights, reported, xs, dt_in, dt_out)
        ex = exact.exact_fedavg(weights, reported, vals)
        assert N == sum(w for w, r in zip(weights, reported) if r)
        assert cnt == sum(reported)
        if ex is None:
            assert out is None
            continue
        if dt_out == "f32":
            want = [exact.nearest_f32(v) for v in ex]
            assert out.view(np.uint32).tolist() == want
        else:
            want = [exact.nearest_bf16(v) for v in ex]
            assert out.tolist() == want


def test_against_numpy_average():
    """The fp64 quotient agrees with numpy.average(weights=...) to fp64 rounding."""
    rng = np.random.default_rng(12)
    K, m = 7, 5000
    weights = rng.integers(1, 5000, K).astype(np.float64)
    xs = [(rng.standard_normal(m) * 0.02).astype(np.float32) for _ in range(K)]
    y = oracle.fedavg_key_f64(weights, [True] * K, xs, "f32")
    ref = np.average(np.stack([x.astype(np.float64) for x in xs]), axis=0, weights=weights)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-18)
    # dropping a client (a "dropped term") must be detectable
    y2 = oracle.fedavg_key_f64(weights, [True] * (K - 1) + [False], xs, "f32")
    assert not np.allclose(y2, ref, rtol=1e-13, atol=1e-18)


# ----------------------------------------------------------------- invariants
def test_single_client_returns_itself():
    rng = np.random.default_rng(13)
    for dt in ("f32", "bf16"):
        x = (rng.standard_normal(4097) * 0.05).astype(np.float32) if dt == "f32" else _random_bf16(rng, 4097, 0.05)
        out, N, cnt = oracle.fedavg_key([873.0], [True], [x], dt, dt)
        assert np.array_equal(out.view(np.uint8), x.view(np.uint8))


def test_identical_clients_return_that_model():
    rng = np.random.default_rng(14)
    for dt in ("f32", "bf16"):
        x = (rng.standard_normal(1000) * 0.02).astype(np.float32) if dt == "f32" else _random_bf16(rng, 1000, 0.02)
        w = [float(v) for v in rng.integers(1, 5000, 9)]
        out, _, _ = oracle.fedavg_key(w, [True] * 9, [x] * 9, dt, dt)
        assert np.array_equal(out.view(np.uint8), x.view(np.uint8))


def test_equal_weights_is_simple_mean():
    """Clara's first case: the simple average of all clients (numpy.mean)."""
    rng = np.random.default_rng(15)
    for K in (2, 4, 8, 5):
        xs = [_random_bf16(rng, 3000, 0.01) for _ in range(K)]
        y = oracle.fedavg_key_f64([250.0] * K, [True] * K, xs, "bf16")
        ref = np.mean(np.stack([_bf16_to_f64(x) for x in xs]), axis=0)
        if K & (K - 1) == 0:
            assert np.array_equal(y, ref)     # all sums exact, division by 2^j exact
        else:
            assert np.allclose(y, ref, rtol=2.3e-16, atol=0)


def test_permutation_invariance_all_orders():
    rng = np.random.default_rng(16)
    K = 4
    xs = [(rng.standard_normal(2000) * 0.05).astype(np.float32) for _ in range(K)]
    w = [float(v) for v in rng.integers(100, 1001, K)]
    base = None
    for perm in itertools.permutations(range(K)):
        out, _, _ = oracle.fedavg_key([w[p] for p in perm], [True] * K, [xs[p] for p in perm], "f32", "f32")
        if base is None:
            base = out
        assert np.array_equal(out, base)


def test_absent_client_contributes_nothing():
    rng = np.random.default_rng(17)
    K = 5
    xs = [(rng.standard_normal(500) * 0.05).astype(np.float32) for _ in range(K)]
    w = [float(v) for v in rng.integers(100, 1001, K)]
    rep = [True, False, True, True, False]
    poisoned = list(xs)
    poisoned[1] = np.full(500, np.nan, np.float32)
    poisoned[4] = np.full(500, np.inf, np.float32)
    a, Na, ca = oracle.fedavg_key(w, rep, poisoned, "f32", "f32")
    keep = [k for k in range(K) if rep[k]]
    b, Nb, cb = oracle.fedavg_key([w[k] for k in keep], [True] * 3, [xs[k] for k in keep], "f32", "f32")
    assert np.array_equal(a, b) and Na == Nb and ca == cb == 3


def test_per_key_denominator_for_partial_reporters():
    """A key sent by one client alone comes back as that client's values, not
    shrunk by the weights of clients that did not send it (client update contract)."""
    x1 = _bf16_bits([0.5, -0.25, 3.0])
    out, N, cnt = oracle.fedavg_key([400.0, 100.0], [False, True], [None, x1], "bf16", "bf16")
    assert out.tolist() == x1.tolist() and N == 100.0 and cnt == 1


def test_no_weight_leaves_key_untouched():
    x = _f32([1.0, 2.0])
    sentinel = np.array([7.0, 7.0], np.float32)
    res, N, cnt = oracle.fedavg_key([0.0, 0.0], [True, True], [x, x], "f32", "f32", out=sentinel)
    assert res is None and N == 0.0 and cnt == 2 and sentinel.tolist() == [7.0, 7.0]
    res, N, cnt = oracle.fedavg_key([5.0, 3.0], [False, False], [x, x], "f32", "f32", out=sentinel)
    assert res is None and N == 0.0 and cnt == 0


def test_zero_weight_reporter_counts_but_adds_nothing():
    x0, x1 = _f32([100.0]), _f32([2.0])
    out, N, cnt = oracle.fedavg_key([0.0, 9.0], [True, True], [x0, x1], "f32", "f32")
    assert out.tolist() == [2.0] and N == 9.0 and cnt == 2


def test_convex_bound():
    rng = np.random.default_rng(18)
    K = 6
    xs = [_random_bf16(rng, 5000, 0.02) for _ in range(K)]
    w = [float(v) for v in rng.integers(1, 5000, K)]
    out, _, _ = oracle.fedavg_key(w, [True] * K, xs, "bf16", "bf16")
    v = np.stack([_bf16_to_f64(x) for x in xs])
    o = _bf16_to_f64(out)
    assert np.all(o >= v.min(axis=0)) and np.all(o <= v.max(axis=0))


def test_scale_invariance():
    rng = np.random.default_rng(19)
    K = 5
    xs = [(rng.standard_normal(3000) * 0.05).astype(np.float32) for _ in range(K)]
    w = [float(v) for v in rng.integers(100, 1001, K)]
    a, _, _ = oracle.fedavg_key(w, [True] * K, xs, "f32", "bf16")
    for j in (-3, 1, 7):
        b, _, _ = oracle.fedavg_key([v * 2.0 ** j for v in w], [True] * K, xs, "f32", "bf16")
        assert np.array_equal(a, b)


def test_nan_propagates():
    x0 = _f32([1.0, np.nan])
    x1 = _f32([3.0, 1.0])
    out, _, _ = oracle.fedavg_key([1.0, 1.0], [True, True], [x0, x1], "f32", "f32")
    assert out[0] == 2.0 and np.isnan(out[1])
