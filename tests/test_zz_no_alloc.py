"""fa_aggregate_noalloc: aggregation of one tensor without any allocation.

It serves callers that cannot let a library call cudaMalloc -- a process whose
device memory belongs to another allocator or that forbids allocation on its
request path -- by keeping the fp32 running sum in a fixed 16 MiB array of the
library.  These tests call it through the C ABI and compare it with the regular
fa_open / fa_accumulate / fa_finalize path on the same inputs: the same kernels in
the same client order, so the same bits, on two calls in a row (the second call runs
over the first call's leftovers in the shared array), with aligned and unaligned
client pointers; and with the fp64 oracle directly.  Its own error word is checked
after the calls.  This file is named to be collected last."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
from tests.compare import check_bf16, check_f32

pytestmark = pytest.mark.gpu


def _host_inputs(rng, K, n, dtype):
    v = [(rng.standard_normal(n) * 0.02).astype(np.float32) for _ in range(K)]
    if dtype == "bf16":
        v = [(a.view(np.uint32) >> 16).astype(np.uint16) for a in v]
    return v


def _inputs(rng, K, n, dtype, offset=0):
    """Device copies; with `offset`, every tensor starts `offset` elements into its
    allocation (an unaligned pointer for offset 1)."""
    host = _host_inputs(rng, K, n, dtype)
    dev = []
    for a in host:
        t = torch.from_numpy(np.concatenate([np.zeros(offset, a.dtype), a]).view(
            np.int16 if dtype == "bf16" else np.float32)).cuda()
        dev.append(t[offset:])
    return host, dev


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


@pytest.mark.parametrize("offset", [0, 1])
def test_same_bits_as_regular_path_two_calls_in_a_row(offset):
    rng = np.random.default_rng(42 + offset)
    cases = [(5, 3_000_017, "bf16", "bf16"), (19, 1_234_567, "f32", "f32")]
    for call, (K, n, din, dout) in enumerate(cases):
        weights = [float(v) for v in rng.integers(100, 5000, K)]
        _, xs = _inputs(rng, K, n, din, offset)
        out = torch.full((n,), 3, dtype=torch.float32 if dout == "f32" else torch.int16, device="cuda")
        fa.fa_aggregate_noalloc(weights, xs, n, din, dout, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        want = _regular(weights, xs, n, din, dout)
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), f"call {call}, offset {offset}"
    fa.fa_aggregate_noalloc_status()


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32")])
def test_matches_the_oracle_at_the_largest_size(din, dout):
    rng = np.random.default_rng(7 if din == "bf16" else 8)
    n = fa.FA_NOALLOC_MAX_ELEMS
    K = 6
    weights = [float(v) for v in rng.integers(100, 1001, K)]
    host, xs = _inputs(rng, K, n, din)
    out = torch.empty(n, dtype=torch.float32 if dout == "f32" else torch.int16, device="cuda")
    fa.fa_aggregate_noalloc(weights, xs, n, din, dout, out)
    torch.cuda.synchronize()
    fa.fa_aggregate_noalloc_status()
    got = out.cpu().numpy()
    want, _, _ = oracle.fedavg_key(weights, [True] * K, host, din, dout)
    if dout == "bf16":
        check_bf16(got.view(np.uint16), want, "noalloc vs oracle")
    else:
        check_f32(got, want, max(float(np.abs(h).max()) for h in host), K, "noalloc vs oracle")


def test_no_device_memory_is_taken():
    rng = np.random.default_rng(7)
    n = 100_000
    _, xs = _inputs(rng, 3, n, "bf16")
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
