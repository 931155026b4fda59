"""fa_accumulate_keys on the GPU: one client's many chunks in one call.  Bit-identical to
the same chunks sent one by one through fa_accumulate (the adapter workload: partial
participation, up to 256 keys per client, so several 48-segment launches per call),
host chunks read in place, the memory-kind rules, all-or-nothing validation, and the
launch count."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
import synth
from synth import workloads as W
from tests.compare import Bf16Tally, fp32_sum_model
from tests.gpu_helpers import sentinel, sentinel_np, to_dev, to_np, to_pinned

pytestmark = pytest.mark.gpu


def _layout(w):
    return [(name, n) for (name, _), n in zip(w.keys, w.numels)]


@pytest.fixture(scope="module")
def lora():
    w = W.make("lora")
    host = {(k, p): synth.client_key(w, k, p) for k in range(w.K) for p in w.reports[k]}
    return w, host


def _round(w, host, mode, split=False, **opts):
    """mode: 'single' (one fa_accumulate per chunk) or a memory kind for one
    fa_accumulate_keys call per client ('device', 'pinned', 'pageable')."""
    ctx = fa.fa_open(_layout(w), w.dtype_in, w.dtype_out, w.K, **opts)
    keep = []
    try:
        s = torch.cuda.current_stream()
        launches0 = fa.fa_get_stats(ctx)["kernel_launches"]
        for k in range(w.K):
            keys, offs, ptrs, lens = [], [], [], []
            for p in w.reports[k]:
                x = host[(k, p)]
                t = to_dev(x) if mode in ("single", "device") else (to_pinned(x) if mode == "pinned" else x.copy())
                keep.append(t)
                n = w.numels[p]
                cuts = [(0, n)] if not split else [(0, n // 3), (n // 3, n)]   # ragged, unaligned
                for a, b in cuts:
                    keys.append(p)
                    offs.append(a)
                    ptrs.append(fa._ptr(t) + a * x.itemsize)
                    lens.append(b - a)
            if mode == "single":
                for key, a, ptr, n in zip(keys, offs, ptrs, lens):
                    fa.fa_accumulate(ctx, k, w.weights[k], key, a, ptr, n, s)
            else:
                try:
                    fa.fa_accumulate_keys(ctx, k, w.weights[k], keys, offs, ptrs, lens, s)
                except fa.FedAvgError as e:
                    if mode == "pageable" and e.status == fa.FA_ERR_ARG:
                        pytest.skip("this device does not read pageable host memory in place")
                    raise
        launches = fa.fa_get_stats(ctx)["kernel_launches"] - launches0
        outs = [sentinel(n, w.dtype_out) for n in w.numels]
        fa.fa_finalize(ctx, outs, s)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        totals = [fa.fa_key_total(ctx, p) for p in range(w.n_keys)]
        stats = fa.fa_get_stats(ctx)
        return [to_np(o, w.dtype_out) for o in outs], totals, launches, stats
    finally:
        fa.fa_close(ctx)


@pytest.mark.parametrize("mode", ["device", "pinned", "pageable"])
@pytest.mark.parametrize("split", [False, True])
def test_keys_call_bit_identical_to_single_calls(lora, mode, split):
    w, host = lora
    ref, ref_totals, ref_launches, _ = _round(w, host, "single", split)
    got, totals, launches, stats = _round(w, host, mode, split)
    assert totals == ref_totals
    for p in range(w.n_keys):
        assert np.array_equal(got[p], ref[p]), f"key {p}"
    # one launch per <= 48 segments of a client's call instead of one per chunk
    segs = [len(w.reports[k]) * (2 if split else 1) for k in range(w.K)]
    assert launches <= sum(-(-n // 48) for n in segs) < ref_launches
    assert stats["chunks"] == sum(segs)
    assert stats["h2d_bytes"] == (0 if mode == "device" else stats["client_bytes"])
    # and the oracle
    tally = Bf16Tally()
    for p in range(w.n_keys):
        rep = [p in set(w.reports[k]) for k in range(w.K)]
        xs = [host.get((k, p)) for k in range(w.K)]
        want, N, cnt = oracle.fedavg_key(w.weights, rep, xs, w.dtype_in, w.dtype_out)
        assert totals[p] == (N, cnt)
        if want is None:
            assert np.array_equal(got[p], sentinel_np(w.numels[p], w.dtype_out))
            continue
        mx = max(float(np.abs(synth.to_f64(xs[k], w.dtype_in)).max()) for k in range(w.K) if rep[k])
        tally.add(got[p], want, f"key {p}", model=fp32_sum_model(w.weights, rep, xs, "bf16"),
                  bound=1e-6 * mx * cnt)
    tally.check("lora via fa_accumulate_keys")


def _f32(rng, n):
    return (rng.standard_normal(n) * 0.05).astype(np.float32)


def test_keys_call_flat_chunks_and_misaligned_pointers():
    """FLAT chunks spanning keys mixed with per-key chunks in one call; chunk pointers at
    odd element offsets (scalar path); fp32 in and out against the oracle."""
    rng = np.random.default_rng(8)
    numels = [4096 * 3 + 5, 17, 9000, 1, 4100]
    offs = np.cumsum([0] + numels)
    P = int(offs[-1])
    K = 2
    xs = [_f32(rng, P) for _ in range(K)]
    w = [3.0, 7.0]
    ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], "f32", "f32", K)
    try:
        d = [to_dev(np.concatenate([np.zeros(1, np.float32), x])) for x in xs]   # +1: misaligned
        base = [t.data_ptr() + 4 for t in d]
        # client 0: flat [0, 12302) + key 2 + flat rest; client 1: per key, in reverse order
        c0 = [(fa.FA_KEY_FLAT, 0, int(offs[2])), (2, 0, numels[2]),
              (fa.FA_KEY_FLAT, int(offs[3]), P - int(offs[3]))]
        fa.fa_accumulate_keys(ctx, 0, w[0], [c[0] for c in c0], [c[1] for c in c0],
                              [base[0] + 4 * (c[1] if c[0] == -1 else int(offs[c[0]]) + c[1]) for c in c0],
                              [c[2] for c in c0])
        c1 = [(p, 0, numels[p]) for p in reversed(range(len(numels)))]
        fa.fa_accumulate_keys(ctx, 1, w[1], [c[0] for c in c1], [c[1] for c in c1],
                              [base[1] + 4 * int(offs[c[0]]) for c in c1], [c[2] for c in c1])
        outs = [sentinel(n, "f32") for n in numels]
        fa.fa_finalize(ctx, outs)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
    finally:
        fa.fa_close(ctx)
    for p, n in enumerate(numels):
        sl = slice(int(offs[p]), int(offs[p + 1]))
        want, _, _ = oracle.fedavg_key(w, [True, True], [x[sl] for x in xs], "f32", "f32")
        mx = max(float(np.abs(x[sl]).max()) for x in xs)
        got = outs[p].cpu().numpy()
        assert np.abs(got.astype(np.float64) - want).max() <= 1e-6 * mx * K, p


def test_keys_call_rules_and_atomicity():
    n = 5000
    rng = np.random.default_rng(9)
    x = [_f32(rng, n) for _ in range(2)]
    ctx = fa.fa_open([("a", n), ("b", n)], "f32", "f32", 2)
    code = lambda *a: _status(fa.fa_accumulate_keys, ctx, *a)
    try:
        d0, h0 = to_dev(x[0]), to_pinned(x[1])
        # a device chunk with a host chunk: refused, nothing recorded
        assert code(0, 2.0, [0, 1], [0, 0], [d0, h0], [n, n]) == fa.FA_ERR_ARG
        # the last chunk past the end: refused, nothing recorded
        assert code(0, 2.0, [0, 1], [0, 1], [d0, d0], [n, n]) == fa.FA_ERR_RANGE
        # two chunks of key a that together exceed it
        assert code(0, 2.0, [0, 0], [0, 0], [d0, d0], [n, 1]) == fa.FA_ERR_RANGE
        assert fa.fa_key_total(ctx, 0) == (0.0, 0) and fa.fa_key_total(ctx, 1) == (0.0, 0)
        assert fa.fa_get_stats(ctx)["chunks"] == 0
        # then the same client sends the right chunks
        fa.fa_accumulate_keys(ctx, 0, 2.0, [0, 1], [0, 0], [d0, d0], [n, n])
        fa.fa_accumulate_keys(ctx, 1, 3.0, [1, 0], [0, 0], [h0, h0], [n, n])
        assert code(1, 4.0, [0], [0], [h0], [1]) == fa.FA_ERR_WEIGHT
        out = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(2)]
        fa.fa_finalize(ctx, out)
        fa.fa_sync(ctx)
        want, _, _ = oracle.fedavg_key([2.0, 3.0], [True, True], x, "f32", "f32")
        for o in out:
            assert np.abs(o.cpu().numpy().astype(np.float64) - want).max() <= 1e-6 * 0.3 * 2
        assert code(0, 2.0, [0], [0], [d0], [1]) == fa.FA_ERR_STATE
    finally:
        fa.fa_close(ctx)
    staged = fa.fa_open([("a", n)], "f32", "f32", 1, flags=fa.FA_STAGE_HOST)
    try:
        assert _status(fa.fa_accumulate_keys, staged, 0, 1.0, [0], [0], [to_pinned(x[0])], [n]) == fa.FA_ERR_ARG
        fa.fa_accumulate_keys(staged, 0, 1.0, [0], [0], [to_dev(x[0])], [n])    # device chunks fine
        fa.fa_accumulate_keys(staged, 0, 1.0, [], [], [], [])                    # empty call: no-op
    finally:
        torch.cuda.synchronize()
        fa.fa_close(staged)


def _status(fn, *args):
    try:
        fn(*args)
        return fa.FA_OK
    except fa.FedAvgError as e:
        return e.status


@pytest.mark.parametrize("kind", ["device", "pageable"])
def test_keys_calls_from_concurrent_threads(lora, kind):
    """Every client sends its list from its own host thread and stream at the same time;
    calls on one context serialize, contributions land in some client order, and the
    result stays within the order-free bound of the oracle with exact totals."""
    import threading
    w, host = lora
    ctx = fa.fa_open(_layout(w), w.dtype_in, w.dtype_out, w.K)
    errors = []
    keep = {}
    for k in range(w.K):
        keep[k] = [to_dev(host[(k, p)]) if kind == "device" else host[(k, p)].copy()
                   for p in w.reports[k]]
    torch.cuda.synchronize()

    def client(k):
        try:
            s = torch.cuda.Stream()
            ps = w.reports[k]
            fa.fa_accumulate_keys(ctx, k, w.weights[k], ps, [0] * len(ps), keep[k],
                                  [w.numels[p] for p in ps], s)
            s.synchronize()
        except fa.FedAvgError as e:
            errors.append(e)

    try:
        th = [threading.Thread(target=client, args=(k,)) for k in range(w.K)]
        for t in th:
            t.start()
        for t in th:
            t.join()
        if errors and kind == "pageable" and all(e.status == fa.FA_ERR_ARG for e in errors):
            pytest.skip("this device does not read pageable host memory in place")
        assert not errors, errors
        outs = [sentinel(n, w.dtype_out) for n in w.numels]
        fa.fa_finalize(ctx, outs)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        for p in range(w.n_keys):
            rep = [p in set(w.reports[k]) for k in range(w.K)]
            xs = [host.get((k, p)) for k in range(w.K)]
            want, N, cnt = oracle.fedavg_key(w.weights, rep, xs, w.dtype_in, w.dtype_out)
            assert fa.fa_key_total(ctx, p) == (N, cnt)
            got = to_np(outs[p], w.dtype_out)
            if want is None:
                assert np.array_equal(got, sentinel_np(w.numels[p], w.dtype_out))
                continue
            from tests.compare import check_f32_to_bf16
            mx = max(float(np.abs(synth.to_f64(xs[k], w.dtype_in)).max()) for k in range(w.K) if rep[k])
            check_f32_to_bf16(got, want, mx, cnt, f"key {p}")
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)
