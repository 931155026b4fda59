"""fa_accumulate_final: the last contribution to a range fused with its finalize.  The
outputs must be the bits of fa_accumulate for that chunk followed by fa_finalize, for every
ingest form the call takes (device memory, pinned and pageable host memory read in place),
every output form (device memory, pinned host memory written in place), every dtype pair
(the bulk kernel's two result slots and the direct kernel for fp32 in / bf16 out), the
compensated mode, unaligned and ragged chunks, flat chunks across keys, and a key finished
partly through final calls and partly through fa_finalize.  And it must refuse what it
cannot do without changing the round.  (The plain path's outputs are checked against the
oracle by the parity tests; the totals are checked against it here.)"""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
import synth
from synth import workloads as W
from tests.gpu_helpers import ragged_splits, sentinel, to_dev, to_np, to_pinned

pytestmark = pytest.mark.gpu


def _layout(numels):
    return [(f"k{i}", n) for i, n in enumerate(numels)]


def _inputs(rng, numels, K, din, scale=0.02):
    xs = []
    for _ in range(K):
        per = []
        for n in numels:
            v = (rng.standard_normal(n) * scale).astype(np.float32)
            per.append(v if din == "f32" else (v.view(np.uint32) >> 16).astype(np.uint16))
        xs.append(per)
    return xs


def _put(x, mode):
    if mode == "device":
        return to_dev(x)
    if mode == "pinned":
        return to_pinned(x)
    return np.ascontiguousarray(x.view(np.int16) if x.dtype == np.uint16 else x)   # pageable


def _outs(numels, dout, where, flat):
    n = sum(numels)
    if flat:
        o = sentinel(n, dout, device="cpu" if where == "pinned" else None)
        return [o.pin_memory() if where == "pinned" else o]
    outs = [sentinel(m, dout, device="cpu" if where == "pinned" else None) for m in numels]
    return [o.pin_memory() for o in outs] if where == "pinned" else outs


def _as_keys(outs, numels, flat, dout):
    if flat:
        a = to_np(outs[0], dout)
        offs = np.cumsum([0] + list(numels))
        return [a[offs[p]:offs[p + 1]] for p in range(len(numels))]
    return [to_np(o, dout) for o in outs]


def _round(numels, din, dout, K, weights, xs, final=False, mode="device", out_where="device",
           flat=False, flags=0, pieces=1, seed=0, offset=0):
    """Clients 0..K-2 per key through fa_accumulate (device memory); client K-1 through
    fa_accumulate_final (or fa_accumulate when final is False) from `mode` memory, in
    `pieces` ragged chunks per key (a flat chunk over the whole layout when flat); then
    fa_finalize.  Returns the outputs per key."""
    rng = np.random.default_rng(seed)
    ctx = fa.fa_open(_layout(numels), din, dout, K, flags=flags | (fa.FA_FLAT_OUT if flat else 0))
    keep = []
    try:
        s = torch.cuda.current_stream()
        outs = _outs(numels, dout, out_where, flat)
        for k in range(K - 1):
            for p, n in enumerate(numels):
                t = to_dev(xs[k][p])
                keep.append(t)
                fa.fa_accumulate(ctx, k, weights[k], p, 0, t, n, s)
        k = K - 1
        call = (lambda *a: fa.fa_accumulate_final(*a[:7], outs, a[7])) if final else fa.fa_accumulate
        if flat:
            x = np.concatenate([xs[k][p] for p in range(len(numels))])
            if offset:
                x = np.concatenate([np.zeros(offset, x.dtype), x])
            t = _put(x, mode)
            keep.append(t)
            base = fa._ptr(t) + offset * x.itemsize
            for a, b in ragged_splits(sum(numels), pieces, rng):
                call(ctx, k, weights[k], fa.FA_KEY_FLAT, a, base + a * x.itemsize, b - a, s)
        else:
            for p, n in enumerate(numels):
                x = xs[k][p]
                if offset:
                    x = np.concatenate([np.zeros(offset, x.dtype), x])
                t = _put(x, mode)
                keep.append(t)
                base = fa._ptr(t) + offset * x.itemsize
                for a, b in ragged_splits(n, pieces, rng):
                    call(ctx, k, weights[k], p, a, base + a * x.itemsize, b - a, s)
        fa.fa_finalize(ctx, outs, s)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        return _as_keys(outs, numels, flat, dout), [fa.fa_key_total(ctx, p) for p in range(len(numels))]
    finally:
        fa.fa_close(ctx)


NUMELS = [7, 8192 * 3 + 5, 1000, 33, 70000, 8, 4096]
PAIRS = [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")]


@pytest.mark.parametrize("din,dout", PAIRS)
@pytest.mark.parametrize("flags", [0, fa.FA_COMPENSATED])
def test_bits_of_accumulate_then_finalize(din, dout, flags):
    rng = np.random.default_rng(11 + len(din) + len(dout) + flags)
    K = 4
    xs = _inputs(rng, NUMELS, K, din)
    weights = [float(v) for v in rng.integers(100, 1000, K)]
    ref, rtot = _round(NUMELS, din, dout, K, weights, xs, final=False, flags=flags)
    for pieces in (1, 3):
        got, gtot = _round(NUMELS, din, dout, K, weights, xs, final=True, flags=flags, pieces=pieces)
        assert gtot == rtot
        for p in range(len(NUMELS)):
            assert np.array_equal(got[p].view(np.uint8), ref[p].view(np.uint8)), (pieces, p)
    # the totals are the oracle's, bit for bit (the plain path's outputs are checked against
    # the oracle by the parity tests; these are its bits)
    for p, n in enumerate(NUMELS):
        _, N, cnt = oracle.fedavg_key(weights, [True] * K, [xs[k][p] for k in range(K)], din, dout)
        assert gtot[p] == (N, cnt)


@pytest.mark.parametrize("mode,out_where", [("device", "pinned"), ("pinned", "device"), ("pinned", "pinned"),
                                            ("pageable", "device")])
@pytest.mark.parametrize("flat", [False, True])
def test_ingest_and_output_forms(mode, out_where, flat):
    rng = np.random.default_rng(7)
    K = 3
    xs = _inputs(rng, NUMELS, K, "bf16")
    weights = [300.0, 700.0, 1000.0]
    ref, rtot = _round(NUMELS, "bf16", "bf16", K, weights, xs, final=False, flat=flat)
    got, gtot = _round(NUMELS, "bf16", "bf16", K, weights, xs, final=True, mode=mode, out_where=out_where,
                       flat=flat, pieces=2)
    assert gtot == rtot
    for p in range(len(NUMELS)):
        assert np.array_equal(got[p], ref[p]), (mode, out_where, flat, p)


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32")])
def test_unaligned_chunks(din, dout):
    rng = np.random.default_rng(3)
    K = 3
    xs = _inputs(rng, NUMELS, K, din)
    weights = [5.0, 9.0, 2.0]
    ref, _ = _round(NUMELS, din, dout, K, weights, xs, final=False)
    got, _ = _round(NUMELS, din, dout, K, weights, xs, final=True, offset=1, pieces=2)
    for p in range(len(NUMELS)):
        assert np.array_equal(got[p].view(np.uint8), ref[p].view(np.uint8)), p


def test_partly_final_then_finalize_the_rest():
    """Client 2 sends the first half of each key through fa_accumulate_final and the second
    half through fa_accumulate; fa_finalize writes the second halves only."""
    rng = np.random.default_rng(5)
    K = 3
    numels = [100, 8192 * 2 + 3, 65]
    xs = _inputs(rng, numels, K, "bf16")
    weights = [1.0, 2.0, 3.0]
    ref, _ = _round(numels, "bf16", "bf16", K, weights, xs, final=False)
    ctx = fa.fa_open(_layout(numels), "bf16", "bf16", K)
    try:
        outs = [sentinel(n, "bf16") for n in numels]
        keep = []
        for k in range(K - 1):
            for p, n in enumerate(numels):
                t = to_dev(xs[k][p])
                keep.append(t)
                fa.fa_accumulate(ctx, k, weights[k], p, 0, t, n)
        for p, n in enumerate(numels):
            t = to_dev(xs[2][p])
            keep.append(t)
            h = n // 2
            fa.fa_accumulate_final(ctx, 2, weights[2], p, 0, t, h, outs)
            torch.cuda.synchronize()
            # the second half is not written yet
            assert np.all(to_np(outs[p], "bf16")[h:] == 0x7FBF)
            fa.fa_accumulate(ctx, 2, weights[2], p, h, t.data_ptr() + h * 2, n - h)
        fa.fa_finalize(ctx, outs)
        fa.fa_sync(ctx)
        for p in range(len(numels)):
            assert np.array_equal(to_np(outs[p], "bf16"), ref[p]), p
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_refusals_leave_the_round_unchanged():
    numels = [64, 64]
    rng = np.random.default_rng(9)
    xs = _inputs(rng, numels, 3, "bf16")
    ctx = fa.fa_open(_layout(numels), "bf16", "bf16", 3, flags=fa.FA_STAGE_HOST)
    try:
        outs = [sentinel(n, "bf16") for n in numels]
        d = [[to_dev(xs[k][p]) for p in range(2)] for k in range(3)]
        fa.fa_accumulate(ctx, 0, 1.0, 0, 0, d[0][0], 32)            # half of key 0

        def expect(status, *args):
            with pytest.raises(fa.FedAvgError) as e:
                fa.fa_accumulate_final(*args)
            assert e.value.status == status, e.value
        expect(fa.FA_ERR_INCOMPLETE, ctx, 1, 2.0, 0, 0, d[1][0], 64, outs)   # client 0 owes half
        fa.fa_accumulate(ctx, 0, 1.0, 0, 32, d[0][0].data_ptr() + 64, 32)
        expect(fa.FA_ERR_ARG, ctx, 1, 2.0, 0, 0, to_pinned(xs[1][0]), 64, outs)  # staged host chunk
        expect(fa.FA_ERR_ARG, ctx, 1, 2.0, 0, 0, d[1][0], 64,
               [torch.zeros(64, dtype=torch.int16), outs[1]])                    # pageable output
        assert fa.fa_key_total(ctx, 0) == (1.0, 1)
        fa.fa_accumulate_final(ctx, 1, 2.0, 0, 0, d[1][0], 64, outs)
        with pytest.raises(fa.FedAvgError) as e:                                 # a new sender
            fa.fa_accumulate(ctx, 2, 4.0, 0, 0, d[2][0], 64)
        assert e.value.status == fa.FA_ERR_STATE
        fa.fa_accumulate(ctx, 2, 4.0, 1, 0, d[2][1], 64)                         # key 1 is open
        base = [sentinel(n, "bf16") for n in numels]
        with pytest.raises(fa.FedAvgError) as e:                                 # plain means
            fa.fa_finalize_apply(ctx, base, outs, 0.5)
        assert e.value.status == fa.FA_ERR_STATE
        torch.cuda.synchronize()
        assert np.all(to_np(outs[1], "bf16") == 0x7FBF)                          # nothing written
        fa.fa_finalize(ctx, outs)
        fa.fa_sync(ctx)
        want0, _, _ = oracle.fedavg_key([1.0, 2.0], [True, True], [xs[0][0], xs[1][0]], "bf16", "bf16")
        want1, _, _ = oracle.fedavg_key([4.0], [True], [xs[2][1]], "bf16", "bf16")
        assert np.all(np.abs(to_np(outs[0], "bf16").astype(np.int32) - want0.astype(np.int32)) <= 1)
        assert np.all(np.abs(to_np(outs[1], "bf16").astype(np.int32) - want1.astype(np.int32)) <= 1)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_full_round_of_a_workload_through_final_calls():
    """The 3-D U-Net workload (fp32, K = 10): the last client through fa_accumulate_final
    in one flat chunk; every element matches the plain round."""
    w = W.make("unet3d")
    xs = [[synth.client_key(w, k, p) for p in range(w.n_keys)] for k in range(w.K)]
    ref, rtot = _round(w.numels, w.dtype_in, w.dtype_out, w.K, w.weights, xs, final=False, flat=True)
    got, gtot = _round(w.numels, w.dtype_in, w.dtype_out, w.K, w.weights, xs, final=True, flat=True)
    assert gtot == rtot
    for p in range(w.n_keys):
        assert np.array_equal(got[p], ref[p]), p


@pytest.mark.slow
def test_last_quotient_is_correctly_rounded_for_every_fp32_sum():
    """The division in the final form, checked exhaustively: for every fp32 bit pattern s as
    the sum before the division (zeros, subnormals, infinities and NaN included) and
    divisors N_p exact in fp32 (powers of two, odd and even integers up to 2^24 - 1, exact
    non-integers), the output is the correctly rounded quotient: the fp64 quotient rounded to
    fp32 (rounding a 53-bit quotient to 24 bits gives the correctly rounded 24-bit quotient).
    Client 0 (weight N_p - 1) sends zeros and client 1 (weight 1) sends s through
    fa_accumulate_final, so its sum is fma(1, s, +0) = s (for s = -0 that is +0, whose
    quotient is +0)."""
    n = 1 << 32
    free, _ = torch.cuda.mem_get_info()
    assert free > 4 * n * 4 + (8 << 30), f"needs about 72 GB free, have {free / 1e9:.0f}"
    S = 1 << 28
    x1 = torch.empty(n, dtype=torch.int32, device="cuda")
    for a in range(0, n, S):
        v = torch.arange(a, a + S, dtype=torch.int64, device="cuda")
        x1[a:a + S] = torch.where(v >= 1 << 31, v - (1 << 32), v).to(torch.int32)
    del v
    x0 = torch.zeros(n, dtype=torch.float32, device="cuda")
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    xs = x1.view(torch.float32)
    neg0 = torch.tensor([0x80000000 - (1 << 32)], dtype=torch.int32, device="cuda")
    ctx = fa.fa_open([("s", n)], "f32", "f32", 2)
    try:
        for d in (1.0, 2.0, 3.0, 7.0, 10.0, 1000.0, 4095.0, 12345.0, 65537.0, 1048575.0, 16777215.0,
                  1.5, 1.75):
            fa.fa_reset(ctx)
            fa.fa_accumulate(ctx, 0, d - 1.0, 0, 0, x0, n)
            fa.fa_accumulate_final(ctx, 1, 1.0, 0, 0, x1, n, [out])
            fa.fa_sync(ctx)
            torch.cuda.synchronize()
            total, _ = fa.fa_key_total(ctx, 0)
            for a in range(0, n, S):
                s = xs[a:a + S]
                want = (s.double() / total).float()
                want = torch.where(x1[a:a + S] == neg0, torch.zeros_like(want), want)
                got = out[a:a + S]
                same = (got.view(torch.int32) == want.view(torch.int32)) | (torch.isnan(got) & torch.isnan(want))
                bad = int((~same).sum())
                assert bad == 0, (d, a, bad)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)
