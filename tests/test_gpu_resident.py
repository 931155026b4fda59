"""fa_reduce_resident: a whole round from resident full updates straight to the
output.  It must give the bits of the streaming path (fa_accumulate of each
update in the same order, then fa_finalize), match the oracle within the
tolerances, and keep the round's bookkeeping exact."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
import synth
from synth import workloads as W
from tests.compare import Bf16Tally, check_f32
from tests.gpu_helpers import sentinel, to_dev, to_np

pytestmark = pytest.mark.gpu


def _flat_inputs(rng, K, P, dtype, sigma=0.02):
    out = []
    for _ in range(K):
        v = (rng.standard_normal(P) * sigma).astype(np.float32)
        out.append(v if dtype == "f32" else (v.view(np.uint32) >> 16).astype(np.uint16))
    return out


def _streamed(layout, din, dout, weights, xs_dev, flags=0):
    P = sum(n for _, n in layout)
    ctx = fa.fa_open(layout, din, dout, len(xs_dev), flags=fa.FA_FLAT_OUT)
    try:
        for k, x in enumerate(xs_dev):
            fa.fa_accumulate(ctx, k, weights[k], fa.FA_KEY_FLAT, 0, x, P)
        out = sentinel(P, dout)
        fa.fa_finalize(ctx, [out])
        torch.cuda.synchronize()
        return to_np(out, dout)
    finally:
        fa.fa_close(ctx)


def _resident(layout, din, dout, weights, xs_dev, per_key=False):
    P = sum(n for _, n in layout)
    K = len(xs_dev)
    ctx = fa.fa_open(layout, din, dout, K, flags=0 if per_key else fa.FA_FLAT_OUT)
    try:
        if per_key:
            outs = [sentinel(n, dout) for _, n in layout]
        else:
            outs = [sentinel(P, dout)]
        fa.fa_reduce_resident(ctx, list(range(K)), weights, xs_dev, outs)
        torch.cuda.synchronize()
        totals = [fa.fa_key_total(ctx, p) for p in range(len(layout))]
        got = np.concatenate([to_np(o, dout) for o in outs])
        return got, totals
    finally:
        fa.fa_close(ctx)


@pytest.mark.parametrize("K", [1, 2, 5, 16, 17, 33])
@pytest.mark.parametrize("din", ["bf16", "f32"])
def test_resident_bit_identical_to_streaming(K, din):
    rng = np.random.default_rng(100 + K)
    numels = [7, 4096 * 5 + 3, 1000, 33, 70000, 8]      # odd sizes: unaligned flat offsets too
    layout = [(f"k{i}", n) for i, n in enumerate(numels)]
    P = sum(numels)
    weights = [float(v) for v in rng.integers(1, 5000, K)]
    xs = [to_dev(x) for x in _flat_inputs(rng, K, P, din)]
    ref = _streamed(layout, din, "f32", weights, xs)
    got, totals = _resident(layout, din, "f32", weights, xs)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    got_k, _ = _resident(layout, din, "f32", weights, xs, per_key=True)
    assert np.array_equal(got_k.view(np.uint32), ref.view(np.uint32))
    assert all(t == (sum(weights), K) for t in totals)
    ref16 = _streamed(layout, din, "bf16", weights, xs)
    got16, _ = _resident(layout, din, "bf16", weights, xs)
    assert np.array_equal(got16, ref16)


@pytest.mark.parametrize("name", ["tiny", "unet3d"])
def test_resident_matches_oracle(name):
    w = W.make(name)
    xs_host = [synth.client_flat(w, k, 0, w.P) for k in range(w.K)]
    xs = [to_dev(x) for x in xs_host]
    got, totals = _resident([(n, m) for (n, _), m in zip(w.keys, w.numels)], w.dtype_in, w.dtype_out,
                            w.weights, xs, per_key=True)
    offs = w.flat_offsets()
    for p, n in enumerate(w.numels):
        sl = slice(offs[p], offs[p] + n)
        want, N, cnt = oracle.fedavg_key(w.weights, [True] * w.K, [x[sl] for x in xs_host],
                                         w.dtype_in, w.dtype_out)
        assert totals[p] == (N, cnt)
        mx = max(float(np.abs(x[sl]).max()) for x in xs_host)
        check_f32(got[sl], want, mx, w.K, f"{name} key {p}")


def test_resident_state_rules():
    rng = np.random.default_rng(7)
    layout = [("a", 100), ("b", 50)]
    xs = [to_dev(x) for x in _flat_inputs(rng, 2, 150, "bf16")]
    ctx = fa.fa_open(layout, "bf16", "bf16", 2, flags=fa.FA_FLAT_OUT)
    try:
        fa.fa_accumulate(ctx, 0, 1.0, 0, 0, xs[0], 10)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_reduce_resident(ctx, [0, 1], [1.0, 2.0], xs, [sentinel(150, "bf16")])
        assert e.value.status == fa.FA_ERR_STATE
        fa.fa_reset(ctx)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_reduce_resident(ctx, [0, 0], [1.0, 2.0], xs, [sentinel(150, "bf16")])
        assert e.value.status == fa.FA_ERR_ARG
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_reduce_resident(ctx, [0, 1], [1.0, -2.0], xs, [sentinel(150, "bf16")])
        assert e.value.status == fa.FA_ERR_WEIGHT
        host = np.zeros(150, np.uint16)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_reduce_resident(ctx, [0, 1], [1.0, 2.0], [xs[0], host], [sentinel(150, "bf16")])
        assert e.value.status == fa.FA_ERR_ARG
        out = sentinel(150, "bf16")
        fa.fa_reduce_resident(ctx, [0, 1], [1.0, 2.0], xs, [out])
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_finalize(ctx, [out])
        assert e.value.status == fa.FA_ERR_STATE
        assert fa.fa_key_total(ctx, 1) == (3.0, 2)
        fa.fa_reset(ctx)
        fa.fa_accumulate(ctx, 1, 4.0, fa.FA_KEY_FLAT, 0, xs[1], 150)
        fa.fa_finalize(ctx, [out])
        torch.cuda.synchronize()
        assert np.array_equal(to_np(out, "bf16"), to_np(xs[1], "bf16"))
    finally:
        fa.fa_close(ctx)
