"""Rounds captured into a CUDA graph and replayed.  A launch-bound round (small tensors,
few clients) costs more in host calls than on the GPU; captured once, a round replays as
one graph launch.  The calls issue only work a graph can replay as it ran (kernels whose
tables ride in their parameters, counters the kernels leave at zero), so every replay over
new contents of the same client buffers must give the bits a fresh round of direct calls
gives; and the calls that need the host during a round refuse to be captured
(FA_ERR_STATE) without spoiling the capture."""
import numpy as np
import pytest
import torch

import server_side_fedavg_gb300 as fa
from tests.gpu_helpers import sentinel, to_np, to_pinned

pytestmark = pytest.mark.gpu

NUMELS = [7, 8192 * 3 + 5, 1000, 33, 70000, 8, 4096]


def _layout(numels):
    return [(f"k{i}", n) for i, n in enumerate(numels)]


def _fill(rng, bufs, din):
    """New client values in the same device buffers (N(0, 0.02); bf16 by truncation)."""
    for b in bufs:
        v = (rng.standard_normal(b.numel()) * 0.02).astype(np.float32)
        if din == "bf16":
            v = (v.view(np.uint32) >> 16).astype(np.uint16).view(np.int16)
        b.copy_(torch.from_numpy(v))


def _bufs(K, n, din):
    dt = torch.float32 if din == "f32" else torch.int16
    return [torch.empty(n, dtype=dt, device="cuda") for _ in range(K)]


def _streamed(ctx, numels, bufs, weights, outs, s, final=False, es=2):
    """Clients in id order, one call per client and key; the last through
    fa_accumulate_final when `final`; then fa_finalize."""
    K = len(bufs)
    offs = np.cumsum([0] + list(numels))
    for k in range(K):
        for p, n in enumerate(numels):
            ptr = bufs[k].data_ptr() + int(offs[p]) * es
            if final and k == K - 1:
                fa.fa_accumulate_final(ctx, k, weights[k], p, 0, ptr, n, outs, s)
            else:
                fa.fa_accumulate(ctx, k, weights[k], p, 0, ptr, n, s)
    fa.fa_finalize(ctx, outs, s)


def _direct(numels, din, dout, bufs, weights, final=False, flags=0):
    """The same round by direct calls on a fresh context: the reference bits."""
    ctx = fa.fa_open(_layout(numels), din, dout, len(bufs), flags=flags)
    try:
        outs = [sentinel(n, dout) for n in numels]
        _streamed(ctx, numels, bufs, weights, outs, None, final, 4 if din == "f32" else 2)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        return [to_np(o, dout) for o in outs]
    finally:
        fa.fa_close(ctx)


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("final", [False, True])
@pytest.mark.parametrize("flags", [0, fa.FA_COMPENSATED])
def test_captured_streamed_round_replays_bit_identical(din, dout, final, flags):
    rng = np.random.default_rng(3)
    K = 4
    weights = [3.0, 17.0, 250.0, 1.0]
    P = sum(NUMELS)
    bufs = _bufs(K, P, din)
    _fill(rng, bufs, din)
    ctx = fa.fa_open(_layout(NUMELS), din, dout, K, flags=flags)
    try:
        outs = [sentinel(n, dout) for n in NUMELS]
        es = 4 if din == "f32" else 2

        def rnd(s):
            fa.fa_reset(ctx)
            _streamed(ctx, NUMELS, bufs, weights, outs, s, final, es)

        # fa_reset waits for the context's work: it runs outside the capture
        s0 = torch.cuda.Stream()
        with torch.cuda.stream(s0):
            rnd(s0)
        torch.cuda.synchronize()
        fa.fa_reset(ctx)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            _streamed(ctx, NUMELS, bufs, weights, outs, torch.cuda.current_stream(), final, es)
        torch.cuda.synchronize()
        for r in range(3):
            _fill(rng, bufs, din)
            for o in outs:
                o.fill_(0x7FBF if dout == "bf16" else -7.0)
            g.replay()
            torch.cuda.synchronize()
            want = _direct(NUMELS, din, dout, bufs, weights, final, flags)
            for p in range(len(NUMELS)):
                assert np.array_equal(to_np(outs[p], dout), want[p]), (r, p)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


@pytest.mark.parametrize("n_keys", [60, 12])
def test_captured_resident_round_replays(n_keys):
    """fa_reduce_resident captured: 60 keys go as one launch with the tables in its
    parameters and a work counter the launch leaves at zero (so every replay hands out all
    the work again); 12 keys as one J-client reduce launch."""
    rng = np.random.default_rng(11)
    numels = [int(x) for x in rng.integers(1, 40000, n_keys)]
    K = 5
    weights = [2.0, 1.0, 7.0, 3.0, 11.0]
    P = sum(numels)
    bufs = _bufs(K, P, "bf16")
    ctx = fa.fa_open(_layout(numels), "bf16", "bf16", K, flags=fa.FA_FLAT_OUT)
    try:
        out = sentinel(P, "bf16")
        ids = list(range(K))

        def rnd(s):
            fa.fa_reduce_resident(ctx, ids, weights, bufs, [out], s)

        _fill(rng, bufs, "bf16")
        s0 = torch.cuda.Stream()
        with torch.cuda.stream(s0):
            rnd(s0)
        torch.cuda.synchronize()
        fa.fa_reset(ctx)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            rnd(torch.cuda.current_stream())
        torch.cuda.synchronize()
        for r in range(4):
            _fill(rng, bufs, "bf16")
            out.fill_(0x7FBF)
            g.replay()
            torch.cuda.synchronize()
            got = to_np(out, "bf16")
            want = np.concatenate(_direct(numels, "bf16", "bf16", bufs, weights))
            assert np.array_equal(got, want), r
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_captured_subset_round_replays():
    """fa_reduce_subsets captured (tables in the launch's parameters): each client sends
    a seeded subset of the keys, packed in its buffer."""
    rng = np.random.default_rng(21)
    n_keys, K = 40, 6
    numels = [int(x) for x in rng.integers(100, 20000, n_keys)]
    weights = [float(x) for x in rng.integers(1, 500, K)]
    keys = [sorted(rng.choice(n_keys, size=int(rng.integers(10, n_keys)), replace=False).tolist())
            for _ in range(K)]
    bufs = [torch.empty(sum(numels[p] for p in ks), dtype=torch.int16, device="cuda") for ks in keys]
    ctx = fa.fa_open(_layout(numels), "bf16", "bf16", K)
    try:
        outs = [sentinel(n, "bf16") for n in numels]

        def rnd(s):
            fa.fa_reduce_subsets(ctx, list(range(K)), weights, bufs, keys, outs, s)

        _fill(rng, bufs, "bf16")
        s0 = torch.cuda.Stream()
        with torch.cuda.stream(s0):
            rnd(s0)
        torch.cuda.synchronize()
        fa.fa_reset(ctx)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            rnd(torch.cuda.current_stream())
        torch.cuda.synchronize()
        for r in range(3):
            _fill(rng, bufs, "bf16")
            for o in outs:
                o.fill_(0x7FBF)
            g.replay()
            torch.cuda.synchronize()
            ref = fa.fa_open(_layout(numels), "bf16", "bf16", K)
            try:
                want = [sentinel(n, "bf16") for n in numels]
                for j in range(K):
                    off = 0
                    for p in keys[j]:
                        fa.fa_accumulate(ref, j, weights[j], p, 0, bufs[j].data_ptr() + 2 * off, numels[p])
                        off += numels[p]
                fa.fa_finalize(ref, want)
                fa.fa_sync(ref)
                torch.cuda.synchronize()
            finally:
                fa.fa_close(ref)
            for p in range(n_keys):
                assert np.array_equal(to_np(outs[p], "bf16"), to_np(want[p], "bf16")), (r, p)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_captured_delta_round_replays():
    """A delta round captured: K clients, then fa_finalize_apply in place onto the model;
    each replay applies the new mean to the model the previous replay left."""
    rng = np.random.default_rng(31)
    K = 3
    weights = [5.0, 1.0, 2.0]
    P = sum(NUMELS)
    bufs = _bufs(K, P, "bf16")
    ctx = fa.fa_open(_layout(NUMELS), "bf16", "bf16", K)
    model = [sentinel(n, "bf16") for n in NUMELS]
    for m in model:
        m.fill_(0x3F80)                     # bf16 1.0
    ref_model = [m.clone() for m in model]
    offs = np.cumsum([0] + NUMELS)
    try:
        def rnd(s):
            for k in range(K):
                for p, n in enumerate(NUMELS):
                    fa.fa_accumulate(ctx, k, weights[k], p, 0, bufs[k].data_ptr() + 2 * int(offs[p]), n, s)
            fa.fa_finalize_apply(ctx, model, model, 0.5, s)

        _fill(rng, bufs, "bf16")
        s0 = torch.cuda.Stream()
        with torch.cuda.stream(s0):
            rnd(s0)
        torch.cuda.synchronize()
        fa.fa_reset(ctx)
        for m, r0 in zip(model, ref_model):
            m.copy_(r0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            rnd(torch.cuda.current_stream())
        torch.cuda.synchronize()
        for r in range(3):
            _fill(rng, bufs, "bf16")
            g.replay()
            ref = fa.fa_open(_layout(NUMELS), "bf16", "bf16", K)
            try:
                for k in range(K):
                    for p, n in enumerate(NUMELS):
                        fa.fa_accumulate(ref, k, weights[k], p, 0, bufs[k].data_ptr() + 2 * int(offs[p]), n)
                fa.fa_finalize_apply(ref, ref_model, ref_model, 0.5)
                fa.fa_sync(ref)
                torch.cuda.synchronize()
            finally:
                fa.fa_close(ref)
            for p in range(len(NUMELS)):
                assert np.array_equal(to_np(model[p], "bf16"), to_np(ref_model[p], "bf16")), (r, p)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_captured_batch_round_replays():
    """fa_accumulate_batch captured: 6 resident clients in one pass per key, then finalize."""
    rng = np.random.default_rng(51)
    K = 6
    weights = [float(x) for x in rng.integers(1, 1000, K)]
    P = sum(NUMELS)
    bufs = _bufs(K, P, "bf16")
    offs = np.cumsum([0] + NUMELS)
    ctx = fa.fa_open(_layout(NUMELS), "bf16", "bf16", K)
    try:
        outs = [sentinel(n, "bf16") for n in NUMELS]

        def rnd(s):
            for p, n in enumerate(NUMELS):
                fa.fa_accumulate_batch(ctx, list(range(K)), weights, p, 0,
                                       [b.data_ptr() + 2 * int(offs[p]) for b in bufs], n, s)
            fa.fa_finalize(ctx, outs, s)

        _fill(rng, bufs, "bf16")
        s0 = torch.cuda.Stream()
        with torch.cuda.stream(s0):
            rnd(s0)
        torch.cuda.synchronize()
        fa.fa_reset(ctx)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            rnd(torch.cuda.current_stream())
        torch.cuda.synchronize()
        for r in range(3):
            _fill(rng, bufs, "bf16")
            for o in outs:
                o.fill_(0x7FBF)
            g.replay()
            torch.cuda.synchronize()
            want = _direct(NUMELS, "bf16", "bf16", bufs, weights)
            for p in range(len(NUMELS)):
                assert np.array_equal(to_np(outs[p], "bf16"), want[p]), (r, p)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_calls_that_need_the_host_refuse_capture():
    """Inside a capture: a staged chunk, a pageable chunk and a pageable output are refused
    with FA_ERR_STATE and issue nothing, so the capture still ends and replays the calls
    that were accepted."""
    numels = [4096, 100]
    K = 2
    P = sum(numels)
    rng = np.random.default_rng(41)
    bufs = _bufs(K, P, "bf16")
    _fill(rng, bufs, "bf16")
    staged = fa.fa_open(_layout(numels), "bf16", "bf16", K, flags=fa.FA_STAGE_HOST)
    ctx = fa.fa_open(_layout(numels), "bf16", "bf16", K)
    host = to_pinned(np.zeros(numels[0], np.uint16))
    pageable = np.zeros(numels[0], np.int16)
    try:
        outs = [sentinel(n, "bf16") for n in numels]
        # a first round outside any capture: every kernel loaded
        for k in range(K):
            fa.fa_accumulate(ctx, k, 1.0, fa.FA_KEY_FLAT, 0, bufs[k], P)
        fa.fa_finalize(ctx, outs)
        fa.fa_sync(ctx)
        fa.fa_reset(ctx)
        torch.cuda.synchronize()

        def refused(call, *args):
            with pytest.raises(fa.FedAvgError) as e:
                call(*args)
            assert e.value.status == fa.FA_ERR_STATE, e.value

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            s = torch.cuda.current_stream()
            refused(fa.fa_accumulate, staged, 0, 1.0, 0, 0, host, numels[0], s)
            refused(fa.fa_accumulate, ctx, 0, 1.0, 0, 0, pageable, numels[0], s)
            for k in range(K):
                fa.fa_accumulate(ctx, k, float(k + 1), fa.FA_KEY_FLAT, 0, bufs[k], P, s)
            refused(fa.fa_finalize, ctx, [torch.zeros(numels[0], dtype=torch.int16), outs[1]], s)
            fa.fa_finalize(ctx, outs, s)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        want = _direct(numels, "bf16", "bf16", bufs, [1.0, 2.0])
        for p in range(len(numels)):
            assert np.array_equal(to_np(outs[p], "bf16"), want[p]), p
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)
        fa.fa_close(staged)
