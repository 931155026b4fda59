"""Device-side wait timeouts, reported per context, made to happen without hanging or
faulting the GPU.

Every mbarrier wait in the pipelined kernels is bounded; one that gives up sets a bit
in its caller's own device error word, the CTA waits (bounded) for the loads it still
has in flight and returns.  FA_TEST_WAIT_EXPIRES makes each CTA's first data wait in
the streaming kernel give up at once, as if its bound had run out, for the first round
of a context.  These tests check that fa_sync then reports FA_ERR_INTERNAL on that
context only, that a second context on the same GPU and the no-allocation entry point
stay clean, and that after fa_reset the next round matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
from tests.compare import check_bf16
from tests.gpu_helpers import to_dev, to_np

pytestmark = pytest.mark.gpu


def _bf16(rng, n, s=0.02):
    return ((rng.standard_normal(n) * s).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _round(ctx, xs, weights, n):
    for k, x in enumerate(xs):
        fa.fa_accumulate(ctx, k, weights[k], 0, 0, x, n)
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    fa.fa_finalize(ctx, [out])
    return out


def test_expired_wait_fails_only_its_own_context_and_recovers():
    rng = np.random.default_rng(5)
    n = 3_000_017                     # several hundred tiles: every CTA of the grid has work
    K = 3
    weights = [300.0, 17.0, 4096.0]
    host = [_bf16(rng, n) for _ in range(K)]
    xs = [to_dev(h) for h in host]
    want, _, _ = oracle.fedavg_key(weights, [True] * K, host, "bf16", "bf16")
    bad = fa.fa_open([("t", n)], "bf16", "bf16", K, flags=fa.FA_TEST_WAIT_EXPIRES)
    good = fa.fa_open([("t", n)], "bf16", "bf16", K)
    try:
        _round(bad, xs, weights, n)
        out_good = _round(good, xs, weights, n)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_sync(bad)
        assert e.value.status == fa.FA_ERR_INTERNAL
        assert "device-side wait" in e.value.detail
        # the other context on the same GPU is not affected
        fa.fa_sync(good)
        torch.cuda.synchronize()
        check_bf16(to_np(out_good, "bf16"), want, "second context")
        # the failed round refuses further work until fa_reset
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_finalize(bad, [torch.empty(n, dtype=torch.int16, device="cuda")])
        assert e.value.status == fa.FA_ERR_CUDA
        fa.fa_reset(bad)
        # the next round runs normally (the test aid covers the first round only)
        out = _round(bad, xs, weights, n)
        fa.fa_sync(bad)
        torch.cuda.synchronize()
        got = to_np(out, "bf16")
        check_bf16(got, want, "round after reset")
        assert np.array_equal(got, to_np(out_good, "bf16"))
    finally:
        torch.cuda.synchronize()
        fa.fa_close(bad)
        fa.fa_close(good)


def test_reset_reports_an_unchecked_expired_wait_and_still_resets():
    rng = np.random.default_rng(6)
    n = 1 << 20
    x = to_dev(_bf16(rng, n))
    ctx = fa.fa_open([("t", n)], "bf16", "bf16", 1, flags=fa.FA_TEST_WAIT_EXPIRES)
    try:
        fa.fa_accumulate(ctx, 0, 5.0, 0, 0, x, n)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_reset(ctx)                   # the discarded round is reported ...
        assert e.value.status == fa.FA_ERR_INTERNAL
        fa.fa_sync(ctx)                        # ... and the word is clear afterwards
        fa.fa_accumulate(ctx, 0, 5.0, 0, 0, x, n)   # the reset happened: a new round
        out = torch.empty(n, dtype=torch.int16, device="cuda")
        fa.fa_finalize(ctx, [out])
        fa.fa_sync(ctx)
        assert torch.equal(out, x)             # one client: the mean is its own update
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_noalloc_status_is_separate_from_contexts():
    """The no-allocation entry point has an error word of its own: clean after normal
    calls, and a context's expired wait does not show up in it."""
    rng = np.random.default_rng(7)
    n = 1 << 20
    xs = [to_dev(_bf16(rng, n)) for _ in range(3)]
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    fa.fa_aggregate_noalloc([1.0, 2.0, 3.0], xs, n, "bf16", "bf16", out)
    fa.fa_aggregate_noalloc([4.0], xs[:1], n, "bf16", "bf16", out)
    fa.fa_aggregate_noalloc_status()
    ctx = fa.fa_open([("t", n)], "bf16", "bf16", 1, flags=fa.FA_TEST_WAIT_EXPIRES)
    try:
        fa.fa_accumulate(ctx, 0, 5.0, 0, 0, xs[0], n)
        torch.cuda.synchronize()
        fa.fa_aggregate_noalloc_status()
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_sync(ctx)
        assert e.value.status == fa.FA_ERR_INTERNAL
        fa.fa_aggregate_noalloc_status()
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)
