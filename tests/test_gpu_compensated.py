"""The compensated mode (FA_COMPENSATED) on the GPU against the oracle.

The running sum is a pair (hi, lo) updated by the Dot2 scheme (error-free product by
fma, Knuth's TwoSum, errors summed into lo), and finalize divides hi + lo with a
remainder-corrected division.  The bf16 rule is held WITHOUT the fp32-sum escape of
the default mode: every element within 1 bf16 ulp of the oracle and >= 99.99 %
bit-identical; fp32 outputs within two fp32 ulps (plus 2^-38 max|x| where the sum
nearly cancels).  Every path (per-key and flat chunks, batches, resident rounds, host
memory read in place, staged) gives the same bits in this mode too.
The divisor pair (N_p above 2^24) and non-integer weights are checked here as well."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
import synth
from synth import workloads as W
from tests.compare import Bf16Tally, bf16_order, check_f32, check_f32_compensated, check_f32_to_bf16
from tests.gpu_helpers import ragged_splits, sentinel, sentinel_np, to_dev, to_np, to_pinned

pytestmark = pytest.mark.gpu

COMP = fa.FA_COMPENSATED


def _vals(rng, n, sigma, dtype):
    v = (rng.standard_normal(n) * sigma).astype(np.float32)
    return v if dtype == "f32" else (v.view(np.uint32) >> 16).astype(np.uint16)


def _f64(x, dtype):
    return synth.to_f64(x, dtype)


def _check_strict(w, host, outs, totals, tally=None):
    """Every key against the oracle: totals exact, unsent keys untouched, bf16 within 1 ulp
    with no escape, fp32 within the compensated bound."""
    own = tally is None
    tally = tally or Bf16Tally()
    worst = 0.0
    for p in range(w.n_keys):
        rep = [p in set(w.reports[k]) for k in range(w.K)]
        xs = [host.get((k, p)) for k in range(w.K)]
        want, N, cnt = oracle.fedavg_key(w.weights, rep, xs, w.dtype_in, w.dtype_out)
        assert totals[p] == (N, cnt), p
        if want is None:
            assert np.array_equal(outs[p], sentinel_np(w.numels[p], w.dtype_out)), p
            continue
        mx = max(float(np.abs(_f64(xs[k], w.dtype_in)).max()) for k in range(w.K) if rep[k])
        if w.dtype_out == "f32":
            worst = max(worst, check_f32_compensated(outs[p], want, mx, f"key {p}"))
        else:
            tally.add(outs[p], want, f"key {p}")
    if own and w.dtype_out == "bf16":
        print(f"{w.name} compensated: {tally.frac():.6%} of {tally.total} bit-identical")
        tally.check(w.name)
    return worst


@pytest.mark.parametrize("name", ["tiny", "unet3d", "lora"])
def test_small_workloads_strict(name):
    from tests.test_gpu_parity import _host_inputs, run_per_key
    w = W.make(name)
    host = _host_inputs(w)
    outs, totals = run_per_key(w, host, flags=COMP)
    worst = _check_strict(w, host, outs, totals)
    print(f"{name} compensated: worst fp32 error {worst:.2f} ulp")


@pytest.mark.parametrize("dout", ["bf16", "f32"])
def test_cancellation_is_exact_to_the_output_rounding(dout):
    """Per element: client 0 sends a, client 1 a tiny b, client 2 -a, weights (3, 1, 3).
    The exact mean is b / 7.  An fp32 running sum loses most of b in 3a + b (the default
    mode lands many ulps away -- its documented limit); the compensated pair keeps it."""
    rng = np.random.default_rng(71)
    n = 200_003
    a = _vals(rng, n, 1.0, "bf16")
    a[a == 0] = 0x3F80                                   # no zero a: keep the cancellation real
    av = _f64(a, "bf16")
    scale = np.exp2(-rng.integers(18, 23, n).astype(np.float64))
    b = oracle.bf16_rne(av * scale * rng.choice([-1.0, 1.0], n) * rng.uniform(1, 2, n))
    neg = a ^ np.uint16(0x8000)
    xs = [a, b, neg]
    weights = [3.0, 1.0, 3.0]
    want, _, _ = oracle.fedavg_key(weights, [True] * 3, xs, "bf16", dout)
    got = {}
    for flags in (0, COMP):
        ctx = fa.fa_open([("t", n)], "bf16", dout, 3, flags=flags)
        try:
            for k in range(3):
                fa.fa_accumulate(ctx, k, weights[k], 0, 0, to_dev(xs[k]), n)
            out = sentinel(n, dout)
            fa.fa_finalize(ctx, [out])
            fa.fa_sync(ctx)
            got[flags] = to_np(out, dout)
        finally:
            fa.fa_close(ctx)
    if dout == "bf16":
        t = Bf16Tally()
        t.add(got[COMP], want, "compensated")
        t.check("compensated cancellation")
        off = np.abs(bf16_order(got[0]) - bf16_order(want)) > 1
    else:
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(want.astype(np.float64)), 1e-38))) - 23)
        # the pair holds b exactly here: within two ulps of b / 7, with no allowance
        assert (np.abs(got[COMP].astype(np.float64) - want) <= 2 * ulp).all()
        off = np.abs(got[0].astype(np.float64) - want) > 2 * ulp
    # the default mode's fp32 sum cannot hold b: most elements land off (its known limit)
    assert off.mean() > 0.5, off.mean()


def _paths(layout, din, dout, weights, xs_host, flags):
    """The same round through every ingest path; returns {path: flat output}."""
    P = sum(n for _, n in layout)
    K = len(xs_host)
    es = xs_host[0].itemsize
    xs = [to_dev(x) for x in xs_host]
    res = {}

    def run(name, body, extra=0):
        ctx = fa.fa_open(layout, din, dout, K, flags=flags | fa.FA_FLAT_OUT | extra)
        try:
            keep = body(ctx)
            out = sentinel(P, dout)
            fa.fa_finalize(ctx, [out])
            fa.fa_sync(ctx)
            torch.cuda.synchronize()
            res[name] = to_np(out, dout)
            del keep
        finally:
            fa.fa_close(ctx)

    def flat(ctx):
        for k in range(K):
            fa.fa_accumulate(ctx, k, weights[k], fa.FA_KEY_FLAT, 0, xs[k], P)

    def ragged(ctx):
        rng = np.random.default_rng(5)
        for k in range(K):
            for a, b in ragged_splits(P, 7, rng):
                fa.fa_accumulate(ctx, k, weights[k], fa.FA_KEY_FLAT, a, xs[k].data_ptr() + a * es, b - a)

    def batch(ctx):
        fa.fa_accumulate_batch(ctx, list(range(K)), weights, fa.FA_KEY_FLAT, 0, xs, P)

    def pinned(ctx):
        hs = [to_pinned(x) for x in xs_host]
        for k in range(K):
            fa.fa_accumulate(ctx, k, weights[k], fa.FA_KEY_FLAT, 0, hs[k], P)
        return hs

    def keys(ctx):
        offs = np.cumsum([0] + [n for _, n in layout])[:-1]
        for k in range(K):
            fa.fa_accumulate_keys(ctx, k, weights[k], list(range(len(layout))), [0] * len(layout),
                                  [xs[k].data_ptr() + int(o) * es for o in offs], [n for _, n in layout])

    run("flat", flat)
    run("ragged", ragged)
    run("batch", batch)
    run("pinned in place", pinned)
    run("pinned staged", pinned, fa.FA_STAGE_HOST)
    run("keys", keys)
    ctx = fa.fa_open(layout, din, dout, K, flags=flags | fa.FA_FLAT_OUT)
    try:
        out = sentinel(P, dout)
        fa.fa_reduce_resident(ctx, list(range(K)), weights, xs, [out])
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        res["resident"] = to_np(out, dout)
    finally:
        fa.fa_close(ctx)
    return res


@pytest.mark.parametrize("K", [3, 16, 19])
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32")])
def test_every_path_gives_the_same_bits(K, din, dout):
    rng = np.random.default_rng(200 + K)
    numels = [7, 6144 * 3 + 5, 1000, 33, 70000, 8, 4096]
    layout = [(f"k{i}", n) for i, n in enumerate(numels)]
    P = sum(numels)
    weights = [float(v) for v in rng.integers(1, 5000, K)]
    xs = [_vals(rng, P, 0.02, din) for _ in range(K)]
    res = _paths(layout, din, dout, weights, xs, COMP)
    ref = res["flat"]
    for name, got in res.items():
        assert np.array_equal(got.view(np.uint8), ref.view(np.uint8)), name
    want, _, _ = oracle.fedavg_key(weights, [True] * K, xs, din, dout)
    if dout == "bf16":
        t = Bf16Tally()
        t.add(ref, want, "compensated")
        t.check("compensated paths")
    else:
        check_f32_compensated(ref, want, max(float(np.abs(x).max()) for x in xs), "compensated paths")


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("lr", [1.0, 0.5])
def test_delta_round_compensated(din, dout, lr):
    rng = np.random.default_rng(41)
    numels = [6144 * 5 + 3, 13, 100_000]
    K = 5
    w = [float(v) for v in rng.integers(100, 1001, K)]
    deltas = [[_vals(rng, n, 1e-3, din) for n in numels] for _ in range(K)]
    base = [_vals(rng, n, 0.02, dout) for n in numels]
    ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], din, dout, K, flags=COMP)
    try:
        for k in range(K):
            for p, n in enumerate(numels):
                fa.fa_accumulate(ctx, k, w[k], p, 0, to_dev(deltas[k][p]), n)
        bases = [to_dev(b) for b in base]
        fa.fa_finalize_apply(ctx, bases, bases, lr)
        torch.cuda.synchronize()
        tally = Bf16Tally()
        for p, n in enumerate(numels):
            want, _, _ = oracle.fedavg_apply_key(w, [True] * K, [deltas[k][p] for k in range(K)], din,
                                                 base[p], lr, dout)
            got = to_np(bases[p], dout)
            if dout == "bf16":
                tally.add(got, want, f"key {p}")
            else:
                # the mean within two ulps, then one rounding of base + lr * mean
                ulp_b = np.exp2(np.floor(np.log2(np.maximum(np.abs(want.astype(np.float64)), 1e-38))) - 23)
                mean = oracle.fedavg_key_f64(w, [True] * K, [deltas[k][p] for k in range(K)], din)
                ulp_m = np.exp2(np.floor(np.log2(np.maximum(np.abs(mean), 1e-38))) - 23)
                d = np.abs(got.astype(np.float64) - want.astype(np.float64))
                assert (d <= ulp_b + 2 * abs(lr) * ulp_m).all(), p
        if dout == "bf16":
            tally.check("compensated delta round")
    finally:
        fa.fa_close(ctx)


@pytest.mark.parametrize("flags", [0, COMP])
@pytest.mark.parametrize("dout", ["bf16", "f32"])
def test_totals_above_2_pow_24(flags, dout):
    """Weights whose per-key total is not exact in fp32 (2^24 + 3, 3 * 2^24 + 1, ...): the
    divisor is a pair of floats.  In the compensated mode identical clients give back their
    update exactly, and other clients match the oracle within its strict bounds.  In the
    default mode, weights with more than 16 significant bits make the products n_k * x
    inexact in fp32, so a bf16 output is held to the fp32 bound plus one bf16 ulp (as for
    fp32 inputs); the fp32 output to the fp32 bound."""
    rng = np.random.default_rng(81)
    n = 50_001
    x = _vals(rng, n, 0.02, "bf16" if dout == "bf16" else "f32")
    din = "bf16" if dout == "bf16" else "f32"
    for weights in ([2.0 ** 24, 1.0, 2.0], [2.0 ** 24] * 3 + [1.0], [2.0 ** 24, 2.0 ** 24 - 3, 2.0 ** 23 + 5, 1.0]):
        K = len(weights)
        # identical clients: the mean is x itself
        ctx = fa.fa_open([("t", n)], din, dout, K, flags=flags)
        try:
            xd = to_dev(x)
            for k in range(K):
                fa.fa_accumulate(ctx, k, weights[k], 0, 0, xd, n)
            out = sentinel(n, dout)
            fa.fa_finalize(ctx, [out])
            fa.fa_sync(ctx)
            assert fa.fa_key_total(ctx, 0) == (sum(weights), K)
            got = to_np(out, dout)
        finally:
            fa.fa_close(ctx)
        if flags & COMP:
            assert np.array_equal(got.view(np.uint8), x.view(np.uint8)), weights
        # different clients, against the oracle
        xs = [_vals(rng, n, 0.02, din) for _ in range(K)]
        ctx = fa.fa_open([("t", n)], din, dout, K, flags=flags)
        try:
            for k in range(K):
                fa.fa_accumulate(ctx, k, weights[k], 0, 0, to_dev(xs[k]), n)
            out = sentinel(n, dout)
            fa.fa_finalize(ctx, [out])
            fa.fa_sync(ctx)
            got = to_np(out, dout)
        finally:
            fa.fa_close(ctx)
        want, _, _ = oracle.fedavg_key(weights, [True] * K, xs, din, dout)
        mx = max(float(np.abs(_f64(v, din)).max()) for v in xs)
        if dout == "f32":
            if flags & COMP:
                check_f32_compensated(got, want, mx, f"{weights}")
            else:
                check_f32(got, want, mx, K, f"{weights}")
        elif flags & COMP:
            t = Bf16Tally()
            t.add(got, want, f"{weights}")
            t.check(f"{weights}")
        else:
            check_f32_to_bf16(got, want, mx, K, f"{weights}")


@pytest.mark.parametrize("flags", [0, COMP])
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32")])
def test_non_integer_weights(flags, din, dout):
    """Weights that are not integers are rounded to fp32 on the device (relative change at
    most 2^-24) while N_p sums them as given: the result stays within the fp32 bound, and
    for bf16 output within the fp32 bound plus one bf16 ulp."""
    rng = np.random.default_rng(91)
    n = 40_000
    weights = [0.37, 12.5, 1e-3, 7.25, 1.0 / 3.0]
    K = len(weights)
    xs = [_vals(rng, n, 0.02, din) for _ in range(K)]
    ctx = fa.fa_open([("t", n)], din, dout, K, flags=flags)
    try:
        for k in range(K):
            fa.fa_accumulate(ctx, k, weights[k], 0, 0, to_dev(xs[k]), n)
        out = sentinel(n, dout)
        fa.fa_finalize(ctx, [out])
        fa.fa_sync(ctx)
        total = fa.fa_key_total(ctx, 0)
        got = to_np(out, dout)
    finally:
        fa.fa_close(ctx)
    want, N, cnt = oracle.fedavg_key(weights, [True] * K, xs, din, dout)
    assert total == (N, cnt)          # summed in client order, as the oracle does
    mx = max(float(np.abs(_f64(v, din)).max()) for v in xs)
    if dout == "f32":
        check_f32(got, want, mx, K, "non-integer weights")
    else:
        check_f32_to_bf16(got, want, mx, K, "non-integer weights")


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32")])
def test_non_finite_values_compensated(din, dout):
    """IEEE propagation holds in the compensated mode too: inf passes through, inf - inf,
    NaN and 0 * inf give NaN, as in the oracle."""
    from tests.test_gpu_edges import _classes
    rng = np.random.default_rng(22)
    n = 3 * 6144 + 7
    K = 3
    w = [3.0, 5.0, 0.0]
    xs = [_vals(rng, n, 0.05, din) for _ in range(K)]
    if din == "f32":
        pinf, ninf, nan = np.float32(np.inf), np.float32(-np.inf), np.float32(np.nan)
    else:
        pinf, ninf, nan = np.uint16(0x7F80), np.uint16(0xFF80), np.uint16(0x7FC0)
    plant = {(0, 10): pinf, (1, 20): nan, (0, 30): pinf, (1, 30): ninf, (2, 40): pinf,
             (0, 50): ninf, (0, 6150): nan, (1, n - 1): pinf}
    for (k, i), v in plant.items():
        xs[k][i] = v
    ctx = fa.fa_open([("k", n)], din, dout, K, flags=COMP)
    try:
        for k in range(K):
            fa.fa_accumulate(ctx, k, w[k], 0, 0, to_dev(xs[k]), n)
        out = sentinel(n, dout)
        fa.fa_finalize(ctx, [out])
        fa.fa_sync(ctx)
        got = to_np(out, dout)
    finally:
        fa.fa_close(ctx)
    want, _, _ = oracle.fedavg_key(w, [True] * K, xs, din, dout)
    as_f = (lambda b: (b.astype(np.uint32) << 16).view(np.float32)) if dout == "bf16" else (lambda a: a)
    assert np.array_equal(_classes(as_f(got)), _classes(as_f(want)))
    fin = _classes(as_f(want)) == 0
    if dout == "bf16":
        t = Bf16Tally()
        t.add(got[fin], want[fin], "finite elements")
    else:
        mx = max(float(np.abs(np.nan_to_num(x, posinf=0, neginf=0)).max()) for x in xs)
        check_f32_compensated(got[fin], want[fin], mx, "finite elements")
