"""fa_aggregate_noalloc: aggregation of one tensor without any allocation.

It serves callers that cannot let a library call cudaMalloc -- a process whose
device memory belongs to another allocator or that forbids allocation on its
request path -- by keeping the fp32 running sum in a fixed 16 MiB array of the
library.  These tests call it through the C ABI and compare it with the regular
fa_open / fa_accumulate / fa_finalize path on the same inputs, within the
tolerances the other parity tests use, on two calls in a row (the second call
runs over the first call's leftovers in the shared array).  This file is named
to be collected last."""
import numpy as np
import pytest
import torch

import server_side_fedavg_gb300 as fa
from tests.compare import check_bf16, check_f32

pytestmark = pytest.mark.gpu


def _inputs(rng, K, n, dtype):
    v = [(rng.standard_normal(n) * 0.02).astype(np.float32) for _ in range(K)]
    if dtype == "bf16":
        v = [(a.view(np.uint32) >> 16).astype(np.uint16).view(np.int16) for a in v]
    return [torch.from_numpy(a).cuda() for a in v]


def _regular(weights, xs, n, din, dout):
    ctx = fa.fa_open([("t", n)], din, dout, len(xs))
    try:
        for k, x in enumerate(xs):
            fa.fa_accumulate(ctx, k, weights[k], 0, 0, x, n)
        out = torch.empty(n, dtype=torch.float32 if dout == "f32" else torch.int16, device="cuda")
        fa.fa_finalize(ctx, [out])
        torch.cuda.synchronize()
        return out.cpu().numpy()
    finally:
        fa.fa_close(ctx)


def test_matches_regular_path_two_calls_in_a_row():
    rng = np.random.default_rng(42)
    cases = [(5, 3_000_017, "bf16", "bf16"), (19, 1_234_567, "f32", "f32")]
    for call, (K, n, din, dout) in enumerate(cases):
        weights = [float(v) for v in rng.integers(100, 5000, K)]
        xs = _inputs(rng, K, n, din)
        out = torch.full((n,), 3, dtype=torch.float32 if dout == "f32" else torch.int16, device="cuda")
        fa.fa_aggregate_noalloc(weights, xs, n, din, dout, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        want = _regular(weights, xs, n, din, dout)
        if dout == "bf16":
            check_bf16(got.view(np.uint16), want.view(np.uint16), f"call {call}")
        else:
            mx = max(float(x.abs().max()) for x in xs)
            check_f32(got, want, mx, K, f"call {call}")


def test_no_device_memory_is_taken():
    rng = np.random.default_rng(7)
    n = 100_000
    xs = _inputs(rng, 3, n, "bf16")
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    fa.fa_aggregate_noalloc([1.0, 2.0, 3.0], xs, n, "bf16", "bf16", out)   # set-up on this device
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        fa.fa_aggregate_noalloc([1.0, 2.0, 3.0], xs, n, "bf16", "bf16", out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_rejects_sizes_beyond_the_array():
    x = torch.zeros(8, dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FedAvgError) as e:
        fa.fa_aggregate_noalloc([1.0], [x], fa.FA_NOALLOC_MAX_ELEMS + 1, "f32", "f32", x)
    assert e.value.status == fa.FA_ERR_RANGE


def test_rejects_inputs_outside_cudamalloc_memory():
    """Inputs are read with bulk copies, so managed and host memory are refused (nothing is
    launched); a managed output, written with plain stores, is accepted."""
    from tests.test_gpu_edges import _managed
    n = 4096
    x = torch.ones(n, dtype=torch.float32, device="cuda")
    mp, mview, free = _managed(n, np.float32)
    try:
        mview[:] = 1.0
        for bad in (mp, np.ones(n, np.float32)):
            with pytest.raises(fa.FedAvgError) as e:
                fa.fa_aggregate_noalloc([1.0], [bad], n, "f32", "f32", x)
            assert e.value.status == fa.FA_ERR_ARG
        mview[:] = -7.0
        fa.fa_aggregate_noalloc([2.0, 6.0], [x, x], n, "f32", "f32", mp)
        torch.cuda.synchronize()
        assert np.all(mview == 1.0)
    finally:
        torch.cuda.synchronize()
        free()
