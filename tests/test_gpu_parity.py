"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small workloads (tiny CNN, 3-D U-Net, LoRA adapters with partial participation)
are compared element by element on every key; the two full-size streamed
workloads (2.2B VLM, 7B decoder) run exactly as bench.py streams them and are
compared on every element (tests/full_compare.py); their other ingest forms
(per key, partial participation, resident, host-fed) on sampled elements the
oracle recomputes one by one.
Tolerances: tests/compare.py."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
import synth
from synth import workloads as W
from tests.compare import Bf16Tally, check_bf16, check_f32, fp32_sum_model
from tests.gpu_helpers import (ragged_splits, sentinel, sentinel_np, to_dev, to_np, to_pinned,
                               torch_dtype)

pytestmark = pytest.mark.gpu


def _layout(w):
    return [(name, n) for (name, _), n in zip(w.keys, w.numels)]


def _host_inputs(w):
    return {(k, p): synth.client_key(w, k, p) for k in range(w.K) for p in w.reports[k]}


def run_per_key(w, host, mode="device", pieces=1, seed=0, **opts):
    """Feed every (client, key) as `pieces` ragged chunks; returns outputs (numpy)."""
    rng = np.random.default_rng(seed)
    if mode.endswith("-staged"):
        opts["flags"] = opts.get("flags", 0) | fa.FA_STAGE_HOST
    ctx = fa.fa_open(_layout(w), w.dtype_in, w.dtype_out, w.K, **opts)
    keep = []
    try:
        s = torch.cuda.current_stream()
        for k in range(w.K):
            for p in w.reports[k]:
                x = host[(k, p)]
                if mode == "device":
                    t = to_dev(x)
                elif mode.startswith("pinned"):
                    t = to_pinned(x)
                else:
                    t = x
                keep.append(t)
                es = x.itemsize
                base = fa._ptr(t)
                for a, b in ragged_splits(w.numels[p], pieces, rng):
                    fa.fa_accumulate(ctx, k, w.weights[k], p, a, base + a * es, b - a, s)
        outs = [sentinel(n, w.dtype_out) for n in w.numels]
        fa.fa_finalize(ctx, outs, s)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        totals = [fa.fa_key_total(ctx, p) for p in range(w.n_keys)]
        return [to_np(o, w.dtype_out) for o in outs], totals
    finally:
        fa.fa_close(ctx)


def check_against_oracle(w, host, outs, totals):
    tally = Bf16Tally()
    for p in range(w.n_keys):
        rep = [p in set(w.reports[k]) for k in range(w.K)]
        xs = [host.get((k, p)) for k in range(w.K)]
        want, N, cnt = oracle.fedavg_key(w.weights, rep, xs, w.dtype_in, w.dtype_out)
        assert totals[p] == (N, cnt), f"key {p}: totals {totals[p]} != oracle {(N, cnt)}"
        if want is None:
            assert np.array_equal(outs[p], sentinel_np(w.numels[p], w.dtype_out)), f"key {p} written"
            continue
        if w.dtype_out == "f32":
            maxw = max(float(np.abs(synth.to_f64(xs[k], w.dtype_in)).max()) for k in range(w.K) if rep[k])
            check_f32(outs[p], want, maxw, cnt, f"key {p}")
        else:
            maxw = max(float(np.abs(synth.to_f64(xs[k], w.dtype_in)).max()) for k in range(w.K) if rep[k])
            tally.add(outs[p], want, f"key {p}", model=fp32_sum_model(w.weights, rep, xs, "bf16"),
                      bound=1e-6 * maxw * cnt)
    if w.dtype_out == "bf16":
        frac = tally.check(w.name)
        print(f"{w.name}: {tally.total} elements, {frac:.6%} bf16 bit-identical")


@pytest.fixture(scope="module")
def small():
    cache = {}

    def get(name):
        if name not in cache:
            w = W.make(name)
            cache[name] = (w, _host_inputs(w))
        return cache[name]
    return get


@pytest.mark.parametrize("name", ["tiny", "unet3d", "lora"])
def test_small_workloads_full_compare(small, name):
    w, host = small(name)
    outs, totals = run_per_key(w, host)
    check_against_oracle(w, host, outs, totals)


def test_lora_has_unreported_modules(small):
    w, _ = small("lora")
    sent = set(p for r in w.reports for p in r)
    # partial participation is exercised: some clients skip modules
    assert any(len(r) < w.n_keys for r in w.reports)
    assert len(sent) <= w.n_keys


@pytest.mark.parametrize("mode", ["device", "pinned", "pinned-staged", "pageable", "pageable-staged"])
@pytest.mark.parametrize("pieces", [1, 5])
def test_ingest_modes_bit_identical(small, mode, pieces):
    """Host (pinned or pageable, read in place by the kernel where the device can address
    it, or through the staging ring) and device ingest, whole or ragged chunks (ragged
    offsets leave pointers unaligned): same bits."""
    w, host = small("lora")
    ref, _ = run_per_key(w, host, "device", 1)
    got, _ = run_per_key(w, host, mode, pieces, seed=3, ring_slots=2, slot_bytes=1 << 20)
    for p in range(w.n_keys):
        assert np.array_equal(got[p], ref[p]), f"key {p}"


def test_ring_geometry_bit_identical(small):
    w, host = small("unet3d")
    a, _ = run_per_key(w, host, "pageable-staged", 3, seed=5, ring_slots=2, slot_bytes=4096)
    b, _ = run_per_key(w, host, "pinned-staged", 1, ring_slots=6, slot_bytes=1 << 24)
    for p in range(w.n_keys):
        assert np.array_equal(a[p], b[p]), f"key {p}"


@pytest.mark.parametrize("J", [2, 3, 8, 11, 16, 19])
def test_batch_bit_identical_to_sequential(J):
    """fa_accumulate_batch == the same clients through fa_accumulate, bit for bit."""
    rng = np.random.default_rng(J)
    numels = [5, 4096 * 3 + 17, 777, 65536]
    layout = [(f"k{i}", n) for i, n in enumerate(numels)]
    weights = [float(v) for v in rng.integers(1, 5000, J)]
    xs = [[to_dev((rng.standard_normal(n) * 0.02).astype(np.float32).view(np.uint32).__rshift__(16).astype(np.uint16))
           for n in numels] for _ in range(J)]
    outs = []
    for batched in (False, True):
        ctx = fa.fa_open(layout, "bf16", "f32", J)
        try:
            for p, n in enumerate(numels):
                if batched:
                    fa.fa_accumulate_batch(ctx, list(range(J)), weights, p, 0, [xs[j][p] for j in range(J)], n)
                else:
                    for j in range(J):
                        fa.fa_accumulate(ctx, j, weights[j], p, 0, xs[j][p], n)
            o = [torch.empty(n, dtype=torch.float32, device="cuda") for n in numels]
            fa.fa_finalize(ctx, o)
            torch.cuda.synchronize()
            outs.append([t.cpu().numpy() for t in o])
        finally:
            fa.fa_close(ctx)
    for p in range(len(numels)):
        assert np.array_equal(outs[0][p].view(np.uint32), outs[1][p].view(np.uint32)), f"key {p}"


def test_flat_chunks_spanning_keys_match_per_key(small):
    """Ragged FLAT chunks across key boundaries == per-key chunks, bit for bit."""
    w, host = small("tiny")
    ref, _ = run_per_key(w, host)
    rng = np.random.default_rng(9)
    ctx = fa.fa_open(_layout(w), w.dtype_in, w.dtype_out, w.K, flags=fa.FA_FLAT_OUT)
    try:
        for k in range(w.K):
            flat = to_dev(synth.client_flat(w, k, 0, w.P))
            for a, b in ragged_splits(w.P, 13, rng):
                fa.fa_accumulate(ctx, k, w.weights[k], fa.FA_KEY_FLAT, a, flat.data_ptr() + a * 4, b - a)
        out = sentinel(w.P, w.dtype_out)
        fa.fa_finalize(ctx, [out])
        torch.cuda.synchronize()
        got = to_np(out, w.dtype_out)
    finally:
        fa.fa_close(ctx)
    offs = w.flat_offsets()
    for p in range(w.n_keys):
        assert np.array_equal(got[offs[p]:offs[p] + w.numels[p]], ref[p]), f"key {p}"


# ------------------------------------------------------------------ full-size streamed
def _sample_indices(w, n_random=200_000, seed=1):
    """Random elements, both ends of every key, every norm key in full, and both sides of
    every chunk seam."""
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, w.P, n_random, dtype=np.int64)]
    for (name, _), off, n in zip(w.keys, w.flat_offsets(), w.numels):
        idx.append(np.arange(off, off + min(n, 64)))
        idx.append(np.arange(off + n - min(n, 64), off + n))
        if "norm" in name:
            idx.append(np.arange(off, off + n))
    ce = w.chunk_elems
    for c in range(ce, w.P, ce):
        idx.append(np.arange(max(0, c - 64), min(w.P, c + 64)))
    idx.append(np.arange(w.P - 256, w.P))
    return np.unique(np.concatenate(idx)).astype(np.uint64)


def _check_sampled(got, xs, w, what, strict=False):
    """bf16 output of a full-size workload against the oracle on sampled elements (clients
    applied in id order, as bench.py streams them), with the fp32 sum model for the rare
    elements where the weighted sum nearly cancels -- or, `strict` (the compensated mode),
    with no such escape."""
    want, N, cnt = oracle.fedavg_key(w.weights, [True] * w.K, xs, w.dtype_in, w.dtype_out)
    if strict:
        return check_bf16(got, want, what)
    maxw = max(float(np.abs(synth.to_f64(x, w.dtype_in)).max()) for x in xs)
    return check_bf16(got, want, what, model=fp32_sum_model(w.weights, [True] * w.K, xs, "bf16"),
                      bound=1e-6 * maxw * w.K)


@pytest.mark.slow
@pytest.mark.parametrize("name,flags,fused", [("vlm2b", 0, False), ("llama7b", 0, False), ("llama7b", 0, True),
                                              ("llama7b", fa.FA_COMPENSATED, False)])
def test_full_size_streamed_every_element(name, flags, fused):
    """The full-size round streamed exactly as bench.py streams it (flat chunks of 64 / 256
    MiB, clients in id order), compared with the oracle on EVERY element, key by key.
    `fused`: the last client through fa_accumulate_final, the bench's timed round; else
    every client through fa_accumulate, then fa_finalize.  Default mode: the bf16 rule
    with the fp32-sum escape; compensated mode (FA_COMPENSATED): the plain rule, no
    escape."""
    import bench
    from tests.full_compare import compare_every_element
    w = W.make(name)
    free, _ = torch.cuda.mem_get_info()
    need = w.P * 2 * 2 + w.P * 4 * (2 if flags else 1) + (8 << 30)
    assert free > need, f"needs {need / 1e9:.0f} GB free, have {free / 1e9:.0f}"
    out = bench.run_streamed_round(w, flags=flags, fused=fused)
    got = out.cpu().numpy().view(np.uint16)
    del out
    torch.cuda.empty_cache()
    compare_every_element(w, got, escape=not flags)


@pytest.mark.slow
def test_full_size_per_key_streamed_sampled():
    """The 7B decoder streamed key by key (one fa_accumulate per client and key: 291 launches
    per client, the 131M-element embedding and head in one launch each) instead of in flat
    chunks, sampled against the oracle."""
    w = W.make("llama7b")
    free, _ = torch.cuda.mem_get_info()
    need = w.P * 2 + w.P * 4 + w.P * 2 + (8 << 30)
    assert free > need, f"needs {need / 1e9:.0f} GB free, have {free / 1e9:.0f}"
    idx = _sample_indices(w, seed=7)
    s = torch.cuda.current_stream()
    x = torch.empty(w.P, dtype=torch.int16, device="cuda")      # one client's update at a time
    out = torch.empty(w.P, dtype=torch.int16, device="cuda")
    ctx = fa.fa_open(_layout(w), w.dtype_in, w.dtype_out, w.K, flags=fa.FA_FLAT_OUT)
    try:
        offs = w.flat_offsets()
        for k in range(w.K):
            synth.client_fill_device(w, k, 0, w.P, x.data_ptr(), s.cuda_stream)
            for p, n in enumerate(w.numels):
                fa.fa_accumulate(ctx, k, w.weights[k], p, 0, x.data_ptr() + 2 * offs[p], n, s)
        fa.fa_finalize(ctx, [out], s)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
    finally:
        fa.fa_close(ctx)
    got = out[torch.from_numpy(idx.astype(np.int64)).cuda()].cpu().numpy().view(np.uint16)
    del x, out
    torch.cuda.empty_cache()
    xs = [synth.client_gather(w, k, idx) for k in range(w.K)]
    frac = _check_sampled(got, xs, w, "llama7b per key")
    print(f"llama7b per key: {idx.size} sampled elements, {frac:.6%} bit-identical")


@pytest.mark.slow
def test_full_size_partial_participation_sampled():
    """The 7B decoder where each client sends a seeded subset of the keys (about 70 %, the
    embedding and head among those skipped by some) and a few keys are sent by nobody: every
    key is divided by its own reporters' total, unsent keys keep the caller's values."""
    w = W.make("llama7b")
    free, _ = torch.cuda.mem_get_info()
    need = w.P * 2 + w.P * 4 + w.P * 2 + (8 << 30)
    assert free > need, f"needs {need / 1e9:.0f} GB free, have {free / 1e9:.0f}"
    rng = np.random.default_rng(17)
    nobody = {5, 100, 200}
    reports = [[p for p in range(w.n_keys) if p not in nobody and rng.random() < 0.7]
               for _ in range(w.K)]
    s = torch.cuda.current_stream()
    x = torch.empty(w.P, dtype=torch.int16, device="cuda")
    out = torch.full((w.P,), 0x7FBF, dtype=torch.int16, device="cuda")
    offs = w.flat_offsets()
    ctx = fa.fa_open(_layout(w), w.dtype_in, w.dtype_out, w.K, flags=fa.FA_FLAT_OUT)
    try:
        for k in range(w.K):
            synth.client_fill_device(w, k, 0, w.P, x.data_ptr(), s.cuda_stream)
            ps = reports[k]
            fa.fa_accumulate_keys(ctx, k, w.weights[k], ps, [0] * len(ps),
                                  [x.data_ptr() + 2 * offs[p] for p in ps], [w.numels[p] for p in ps], s)
            s.synchronize()          # x is refilled for the next client
        fa.fa_finalize(ctx, [out], s)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        totals = [fa.fa_key_total(ctx, p) for p in range(w.n_keys)]
    finally:
        fa.fa_close(ctx)
    idx = _sample_indices(w, seed=9).astype(np.int64)
    got = out[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint16)
    del x, out
    torch.cuda.empty_cache()
    key_of = np.searchsorted(np.asarray(offs, np.int64), idx, side="right") - 1
    tally = Bf16Tally()
    for p in np.unique(key_of):
        sel = key_of == p
        ii = idx[sel].astype(np.uint64)
        rep = [p in set(reports[k]) for k in range(w.K)]
        xs = [synth.client_gather(w, k, ii) if rep[k] else None for k in range(w.K)]
        want, N, cnt = oracle.fedavg_key(w.weights, rep, xs, w.dtype_in, w.dtype_out)
        assert totals[p] == (N, cnt), p
        if want is None:
            assert p in nobody and np.all(got[sel] == 0x7FBF), p
            continue
        mx = max(float(np.abs(synth.to_f64(xs[k], w.dtype_in)).max()) for k in range(w.K) if rep[k])
        tally.add(got[sel], want, f"key {p}", model=fp32_sum_model(w.weights, rep, xs, "bf16"),
                  bound=1e-6 * mx * cnt)
    frac = tally.check("llama7b partial")
    print(f"llama7b partial participation: {idx.size} sampled elements, {frac:.6%} bit-identical")


@pytest.mark.slow
@pytest.mark.parametrize("name,flags", [("vlm2b", 0), ("llama7b", 0), ("llama7b", fa.FA_COMPENSATED)])
def test_full_size_resident_sampled(name, flags):
    """fa_reduce_resident over every client's full update resident in HBM (the bench's
    `resident` configuration), sampled against the oracle (compensated mode: the plain
    bf16 rule, no escape)."""
    import bench
    w = W.make(name)
    free, _ = torch.cuda.mem_get_info()
    need = w.K * w.P * 2 + w.P * 2 + w.P * 4 * (2 if flags else 1) + (8 << 30)
    if free < need:
        pytest.fail(f"needs {need / 1e9:.0f} GB free, have {free / 1e9:.0f}")
    idx = _sample_indices(w, seed=2)
    out = bench.run_resident_round(w, flags=flags)
    got = out[torch.from_numpy(idx.astype(np.int64)).cuda()].cpu().numpy().view(np.uint16)
    assert bool(torch.isfinite(out.view(torch.bfloat16)).all())
    del out
    torch.cuda.empty_cache()
    xs = [synth.client_gather(w, k, idx) for k in range(w.K)]
    what = name + " resident" + (" compensated" if flags else "")
    frac = _check_sampled(got, xs, w, what, strict=bool(flags))
    print(f"{what}: {idx.size} sampled elements, {frac:.6%} bit-identical")


@pytest.mark.slow
@pytest.mark.parametrize("name,staged,host_out", [("vlm2b", False, False), ("vlm2b", True, False),
                                                  ("llama7b", False, True)])
def test_full_size_host_fed_sampled(name, staged, host_out):
    """A full-size workload streamed client by client from PINNED HOST memory in its flat
    chunks -- read in place by the kernel over the host link, or through the library's
    staging ring (FA_STAGE_HOST) -- and, for the 7B decoder as bench.py's end-to-end run
    does it, the aggregate written in place into a pinned host buffer; sampled against
    the oracle."""
    w = W.make(name)
    idx = _sample_indices(w, seed=3)
    host = torch.empty(w.P, dtype=torch.int16).pin_memory()
    hv = host.numpy().view(np.uint16)
    flags = fa.FA_FLAT_OUT | (fa.FA_STAGE_HOST if staged else 0)
    ctx = fa.fa_open(_layout(w), w.dtype_in, w.dtype_out, w.K, flags=flags)
    try:
        s = torch.cuda.current_stream()
        for k in range(w.K):
            synth.client_flat(w, k, 0, w.P, out=hv)
            for c0 in range(0, w.P, w.chunk_elems):
                n = min(w.chunk_elems, w.P - c0)
                fa.fa_accumulate(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0, host.data_ptr() + 2 * c0, n, s)
            s.synchronize()              # the pinned buffer is read on `s`: wait before refilling it
        if host_out:
            out = host                   # the input buffer is free now: reuse it as the output
            out.fill_(0x7FBF)
        else:
            out = torch.empty(w.P, dtype=torch.int16, device="cuda")
        fa.fa_finalize(ctx, [out], s)
        fa.fa_sync(ctx)
        s.synchronize()
        st = fa.fa_get_stats(ctx)
        assert st["h2d_bytes"] == w.K * w.P * 2
        assert st["d2h_bytes"] == (w.P * 2 if host_out else 0)
    finally:
        fa.fa_close(ctx)
    if host_out:
        got = hv[idx.astype(np.int64)].copy()
        # the sentinel is a NaN pattern and every aggregate is finite: all P elements written
        assert not np.any((hv & 0x7F80) == 0x7F80), "an output element is not finite (or not written)"
    else:
        got = out[torch.from_numpy(idx.astype(np.int64)).cuda()].cpu().numpy().view(np.uint16)
    del host
    xs = [synth.client_gather(w, k, idx) for k in range(w.K)]
    what = f"{name} host-fed " + ("staged" if staged else "in place") + (", host output" if host_out else "")
    frac = _check_sampled(got, xs, w, what)
    print(f"{what}: {idx.size} sampled elements, {frac:.6%} bit-identical")
