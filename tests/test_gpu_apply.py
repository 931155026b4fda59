"""Delta rounds on the GPU (fa_finalize_apply) against the oracle:
out = round(base + server_lr * weighted mean of the client deltas), per key,
with partial participation, in place and out of place."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
from tests.compare import Bf16Tally, check_f32
from tests.gpu_helpers import sentinel, to_dev, to_np

pytestmark = pytest.mark.gpu


def _vals(rng, n, sigma, dtype):
    v = (rng.standard_normal(n) * sigma).astype(np.float32)
    return v if dtype == "f32" else (v.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("lr", [1.0, 0.5])
@pytest.mark.parametrize("in_place", [False, True])
def test_delta_round_matches_oracle(din, dout, lr, in_place):
    rng = np.random.default_rng(31)
    numels = [4096 * 7 + 5, 13, 100_000, 4096]
    K = 6
    w = [float(v) for v in rng.integers(100, 1001, K)]
    deltas = [[_vals(rng, n, 1e-3, din) for n in numels] for _ in range(K)]
    base = [_vals(rng, n, 0.02, dout) for n in numels]
    reports = [[p for p in range(len(numels)) if (k + p) % 3 != 0] for k in range(K)]
    reports[0] = reports[0] + [3]
    reports = [sorted(set(r) - ({3} if k else set())) for k, r in enumerate(reports)]
    ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], din, dout, K)
    try:
        for k in range(K):
            for p in reports[k]:
                fa.fa_accumulate(ctx, k, w[k], p, 0, to_dev(deltas[k][p]), numels[p])
        bases = [to_dev(b) for b in base]
        outs = bases if in_place else [sentinel(n, dout) for n in numels]
        fa.fa_finalize_apply(ctx, bases, outs, lr)
        torch.cuda.synchronize()
        tally = Bf16Tally()
        for p, n in enumerate(numels):
            rep = [p in reports[k] for k in range(K)]
            want, N, cnt = oracle.fedavg_apply_key(w, rep, [deltas[k][p] for k in range(K)], din,
                                                   base[p], lr, dout)
            got = to_np(outs[p], dout)
            if want is None:
                expect = base[p] if in_place else to_np(sentinel(n, dout), dout)
                assert np.array_equal(got, expect), f"key {p} was written"
            elif dout == "f32":
                mx = max(float(np.abs(deltas[k][p]).max()) for k in range(K) if rep[k])
                # fp32 bound of the mean, scaled by lr, plus one rounding of the sum with the base
                tol_extra = 2.0 ** -23 * float(np.abs(want).max())
                check_f32(got, want, abs(lr) * mx + tol_extra / (1e-6 * cnt), cnt, f"key {p}")
            else:
                tally.add(got, want, f"key {p}")
        if dout == "bf16":
            tally.check("delta round")
    finally:
        fa.fa_close(ctx)


def test_zero_server_lr_returns_base():
    rng = np.random.default_rng(32)
    n = 50_000
    base = _vals(rng, n, 0.02, "bf16")
    ctx = fa.fa_open([("w", n)], "bf16", "bf16", 2)
    try:
        for k in range(2):
            fa.fa_accumulate(ctx, k, 100.0 + k, 0, 0, to_dev(_vals(rng, n, 1e-3, "bf16")), n)
        out = sentinel(n, "bf16")
        fa.fa_finalize_apply(ctx, [to_dev(base)], [out], 0.0)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(out, "bf16"), base)
    finally:
        fa.fa_close(ctx)


def test_apply_rejects_host_base():
    n = 64
    ctx = fa.fa_open([("w", n)], "f32", "f32", 1)
    try:
        fa.fa_accumulate(ctx, 0, 1.0, 0, 0, to_dev(np.ones(n, np.float32)), n)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_finalize_apply(ctx, [np.zeros(n, np.float32)], [sentinel(n, "f32")], 1.0)
        assert e.value.status == fa.FA_ERR_ARG
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_finalize_apply(ctx, [sentinel(n, "f32")], [sentinel(n, "f32")], float("inf"))
        assert e.value.status == fa.FA_ERR_ARG
    finally:
        fa.fa_close(ctx)
