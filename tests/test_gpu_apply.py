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


@pytest.mark.slow
def test_full_size_delta_round_sampled():
    """The 2.2B VLM as a delta round: 8 clients streamed in its 64 MiB flat chunks, then
    fa_finalize_apply(server_lr = 0.5) onto a base model, sampled against the oracle.  The
    bound is the fp32 running-sum bound scaled by server_lr plus one bf16 ulp, and at least
    99.99 % of the sampled elements must be bit-identical."""
    import synth
    from synth import workloads as W
    from tests.compare import check_f32_to_bf16
    w = W.make("vlm2b")
    free, _ = torch.cuda.mem_get_info()
    need = w.K * w.P * 2 + 2 * w.P * 2 + w.P * 4 + (8 << 30)
    if free < need:
        pytest.fail(f"needs {need / 1e9:.0f} GB free, have {free / 1e9:.0f}")
    lr = 0.5
    s = torch.cuda.current_stream()
    bufs = [torch.empty(w.P, dtype=torch.int16, device="cuda") for _ in range(w.K)]
    for k in range(w.K):
        synth.client_fill_device(w, k, 0, w.P, bufs[k].data_ptr(), s.cuda_stream)
    base = torch.empty(w.P, dtype=torch.int16, device="cuda")
    synth.fill_device(w.seed, w.K, 0, w.sigma, "bf16", 0, w.P, base.data_ptr(), s.cuda_stream)
    out = torch.empty(w.P, dtype=torch.int16, device="cuda")
    ctx = fa.fa_open([(n, k) for (n, _), k in zip(w.keys, w.numels)], "bf16", "bf16", w.K,
                     flags=fa.FA_FLAT_OUT)
    try:
        for k in range(w.K):
            for c0 in range(0, w.P, w.chunk_elems):
                n = min(w.chunk_elems, w.P - c0)
                fa.fa_accumulate(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0,
                                 bufs[k].data_ptr() + 2 * c0, n, s)
        fa.fa_finalize_apply(ctx, [base], [out], lr, s)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
    finally:
        fa.fa_close(ctx)
    rng = np.random.default_rng(4)
    idx = np.unique(np.concatenate([rng.integers(0, w.P, 300_000), np.arange(w.P - 300, w.P)]))
    got = out[torch.from_numpy(idx.astype(np.int64)).cuda()].cpu().numpy().view(np.uint16)
    del bufs, base, out
    torch.cuda.empty_cache()
    xs = [synth.client_gather(w, k, idx.astype(np.uint64)) for k in range(w.K)]
    b = synth.gather(w.seed, w.K, 0, w.sigma, "bf16", idx.astype(np.uint64))
    want, _, _ = oracle.fedavg_apply_key(w.weights, [True] * w.K, xs, "bf16", b, lr, "bf16")
    mx = max(float(np.abs(synth.to_f64(x, "bf16")).max()) for x in xs)
    differ = check_f32_to_bf16(got, want, lr * mx, w.K, "vlm2b delta round")
    assert differ <= 1e-4 * idx.size, f"{differ} of {idx.size} sampled elements not bit-identical"
    print(f"vlm2b delta round: {idx.size} sampled, {1 - differ / idx.size:.6%} bit-identical")
