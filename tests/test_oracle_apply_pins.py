"""Pins for the oracle's delta-round step (base + server_lr * weighted mean):
hand sums, exact rational arithmetic, and its reductions to the plain weighted
mean (base = 0, lr = 1) and to the base itself (lr = 0)."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals):
    a = np.asarray(vals, dtype=np.float32)
    assert np.all((a.view(np.uint32) & 0xFFFF) == 0)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _rows():
    out = []
    for line in open(os.path.join(GOLDEN, "apply_hand_sums.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        w, d, b, lr, e = [p.strip() for p in line.split("|")]
        out.append(([float(t) for t in w.split()], [[float(t) for t in c.split()] for c in d.split(";")],
                    [float(t) for t in b.split()], float(lr), [float(t) for t in e.split()]))
    return out


@pytest.mark.parametrize("row", _rows())
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_apply_hand_sums(row, dt):
    w, ds, b, lr, e = row
    conv = (lambda v: np.asarray(v, np.float32)) if dt == "f32" else _bf16
    out, N, cnt = oracle.fedavg_apply_key(w, [True] * len(w), [conv(d) for d in ds], dt, conv(b), lr, dt)
    got = out.astype(np.float64) if dt == "f32" else (out.astype(np.uint32) << 16).view(np.float32)
    assert [float(v) for v in got] == e


def test_apply_exact_rational():
    rng = np.random.default_rng(21)
    for trial in range(40):
        K = int(rng.integers(1, 6))
        m = 12
        w = [float(v) for v in rng.integers(0, 3000, K)]
        rep = [bool(v) for v in rng.integers(0, 2, K)]
        rep[0] = True
        if w[0] == 0:
            w[0] = 1.0
        xs = [(rng.standard_normal(m) * 1e-3).astype(np.float32) for _ in range(K)]
        base = (rng.standard_normal(m) * 0.02).astype(np.float32)
        lr = float(rng.choice([1.0, 0.5, 2.0, 0.1]))
        for dout in ("f32", "bf16"):
            b = base if dout == "f32" else (base.view(np.uint32) >> 16).astype(np.uint16)
            bv = b.astype(np.float64) if dout == "f32" else (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            out, N, cnt = oracle.fedavg_apply_key(w, rep, xs, "f32", b, lr, dout)
            mean = exact.exact_fedavg(w, rep, [x.astype(np.float64).tolist() for x in xs])
            # lr is an fp64 value: the exact target uses that value, not its decimal
            ys = [Fraction(float(bv[i])) + Fraction(lr) * mean[i] for i in range(m)]
            if dout == "f32":
                assert out.view(np.uint32).tolist() == [exact.nearest_f32(y) for y in ys]
            else:
                assert out.tolist() == [exact.nearest_bf16(y) for y in ys]


def test_apply_reduces_to_plain_mean_and_to_base():
    rng = np.random.default_rng(22)
    K, m = 5, 2000
    w = [float(v) for v in rng.integers(100, 1001, K)]
    xs = [(rng.standard_normal(m) * 0.02).astype(np.float32) for _ in range(K)]
    zero = np.zeros(m, np.float32)
    a, _, _ = oracle.fedavg_apply_key(w, [True] * K, xs, "f32", zero, 1.0, "f32")
    b, _, _ = oracle.fedavg_key(w, [True] * K, xs, "f32", "f32")
    assert np.array_equal(a, b)
    base = (rng.standard_normal(m) * 0.02).astype(np.float32)
    c, _, _ = oracle.fedavg_apply_key(w, [True] * K, xs, "f32", base, 0.0, "f32")
    assert np.array_equal(c, base)


def test_apply_leaves_unweighted_key_untouched():
    x = np.ones(4, np.float32)
    sentinel = np.full(4, 9.0, np.float32)
    res, N, cnt = oracle.fedavg_apply_key([0.0], [True], [x], "f32", np.zeros(4, np.float32), 1.0, "f32", out=sentinel)
    assert res is None and sentinel.tolist() == [9.0] * 4
