"""Randomised rounds on the GPU against the oracle.

One context runs several rounds (fa_reset between them).  Each round mixes, in a
shuffled call order: a random subset of keys per client (partial participation,
including clients that send nothing), ragged chunks of each key, every ingest kind
(device memory; pinned and pageable host memory, read in place or through a small
staging ring), FLAT chunks that span key boundaries, a fa_accumulate_batch group
over part of one key, and clients that send all their chunks in one
fa_accumulate_keys call.

The GPU applies contributions in call order and the oracle sums in client-id order
(the arrival-order reading of FedAvg's weighted mean), so outputs are compared with
the order-free bounds: fp32 within 1e-6 * max|w| * K, bf16 within that bound plus
one bf16 ulp.  Weight totals and reporter counts are exact; keys with no weight keep
the caller's values."""
import random

import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
from tests.compare import check_f32, check_f32_to_bf16
from tests.gpu_helpers import sentinel, sentinel_np, to_dev, to_np, to_pinned

pytestmark = pytest.mark.gpu

SIZES = [1, 3, 8, 31, 257, 4096, 4100, 9000, 12289, 70000]
KINDS = ["device", "pinned", "pageable"]


def _values(rng, n, dtype):
    v = (rng.standard_normal(n) * 0.03).astype(np.float32)
    return v if dtype == "f32" else (v.view(np.uint32) >> 16).astype(np.uint16)


def _as_f32(x, dtype):
    return (x.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else x


def _put(x, kind, keep):
    """Pointer to a copy of x in device, pinned or pageable memory (kept alive in `keep`)."""
    if kind == "device":
        t = to_dev(x)
    elif kind == "pinned":
        t = to_pinned(x)
    else:
        t = np.ascontiguousarray(x.copy())
    keep.append(t)
    return fa._ptr(t)


def _cuts(rng, n, most):
    """Ragged split points of [0, n): 1..most+1 pieces."""
    inner = {rng.randrange(1, n) for _ in range(rng.randint(0, most))} if n > 1 else set()
    b = sorted(inner | {0, n})
    return list(zip(b[:-1], b[1:]))


def _plan(rng, numels, K):
    """Per round: reports[k] (sorted key ids), the batch (key, clients, ranges) or None,
    the flat-mode clients, and the shuffled list of single-chunk calls."""
    n_keys = len(numels)
    offs = [0]
    for n in numels:
        offs.append(offs[-1] + n)
    reports = []
    for _ in range(K):
        r = rng.random()
        if r < 0.35:
            reports.append(list(range(n_keys)))
        elif r < 0.45:
            reports.append([])
        else:
            reports.append(sorted(rng.sample(range(n_keys), rng.randint(1, n_keys))))
    full = [k for k in range(K) if len(reports[k]) == n_keys]
    batch = None
    if len(full) >= 2 and rng.random() < 0.8:
        p = rng.randrange(n_keys)
        ks = rng.sample(full, rng.randint(2, len(full)))
        batch = (p, ks, _cuts(rng, numels[p], 2))
    in_batch = set(batch[1]) if batch else set()
    flat = [k for k in full if k not in in_batch and rng.random() < 0.5]
    calls = []
    grouped = []     # clients whose chunks go in one fa_accumulate_keys call
    for k in range(K):
        if k in flat:
            for a, b in _cuts(rng, offs[-1], 5):                 # spans keys
                calls.append((k, fa.FA_KEY_FLAT, a, b, offs[0] + a))
            continue
        mine = []
        for p in reports[k]:
            if batch and p == batch[0] and k in in_batch:
                continue
            for a, b in _cuts(rng, numels[p], 3):
                mine.append((k, p, a, b, offs[p] + a))
        if mine and rng.random() < 0.3:
            rng.shuffle(mine)
            grouped.append((k, mine))
        else:
            calls += mine
    return offs, reports, batch, calls, grouped


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32"), ("f32", "bf16")])
def test_random_rounds(din, dout):
    _random_rounds(din, dout, {"bf16bf16": 11, "f32f32": 12, "bf16f32": 13, "f32bf16": 14}[din + dout])


@pytest.mark.slow
@pytest.mark.parametrize("seed", range(101, 109))
def test_random_rounds_more_seeds(seed):
    pairs = [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32"), ("f32", "bf16")]
    _random_rounds(*pairs[seed % 4], seed)


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32"), ("f32", "bf16")])
def test_random_rounds_with_final_contributions(din, dout):
    """As test_random_rounds, and for each key one client that sends it in per-key chunks
    sends them last, through fa_accumulate_final: those chunks' outputs come from the
    accumulate kernels, the rest of the layout from fa_finalize."""
    _random_rounds(din, dout, {"bf16bf16": 31, "f32f32": 32, "bf16f32": 33, "f32bf16": 34}[din + dout],
                   final=True)


def _random_rounds(din, dout, seed, final=False):
    rng_py = random.Random(seed)
    rng = np.random.default_rng(seed)
    numels = [rng_py.choice(SIZES) for _ in range(9)]
    K = 7
    # odd seeds send host chunks through the staging ring, even ones read them in place
    ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], din, dout, K,
                     ring_slots=3, slot_bytes=64 << 10, flags=fa.FA_STAGE_HOST if seed % 2 else 0)
    s = torch.cuda.Stream()
    try:
        for rnd in range(5):
            offs, reports, batch, calls, grouped = _plan(rng_py, numels, K)
            weights = [float(rng_py.choice([0, 1, 7, 250, 3000, rng_py.randint(1, 1 << 14)]))
                       for _ in range(K)]
            data = [_values(rng, offs[-1], din) for _ in range(K)]   # client k's flat update
            ops = [("one",) + c for c in calls] + [("keys", k, mine) for k, mine in grouped]
            if batch:
                p, ks, ranges = batch
                ops += [("batch", p, ks, a, b) for a, b in ranges]
            rng_py.shuffle(ops)
            if final:
                # per key, one client's per-key chunks move to the end as final contributions
                last = []
                for p in range(len(numels)):
                    cands = sorted({op[1] for op in ops if op[0] == "one" and op[2] == p})
                    if not cands:
                        continue
                    k = rng_py.choice(cands)
                    mine = [op for op in ops if op[0] == "one" and op[1] == k and op[2] == p]
                    ops = [op for op in ops if op not in mine]
                    last += [("final",) + op[1:] for op in mine]
                rng_py.shuffle(last)
                ops += last
            outs = [sentinel(n, dout) for n in numels]
            keep = []
            for op in ops:
                if op[0] == "batch":
                    _, p, ks, a, b = op
                    ptrs = [_put(data[k][offs[p] + a:offs[p] + b], "device", keep) for k in ks]
                    fa.fa_accumulate_batch(ctx, ks, [weights[k] for k in ks], p, a, ptrs, b - a, s)
                elif op[0] == "keys":
                    _, k, mine = op
                    # one memory kind per call; host chunks only where they are read in place
                    kind = "device" if seed % 2 else rng_py.choice(KINDS)
                    args = ([c[1] for c in mine], [c[2] for c in mine], None, [c[3] - c[2] for c in mine])
                    ptrs = [_put(data[k][g:g + (b - a)], kind, keep) for (_, _, a, b, g) in mine]
                    try:
                        fa.fa_accumulate_keys(ctx, k, weights[k], args[0], args[1], ptrs, args[3], s)
                    except fa.FedAvgError as e:
                        # a host without in-place pageable reads refuses the list, recording
                        # nothing: send it from device memory instead
                        assert e.status == fa.FA_ERR_ARG and kind == "pageable", e
                        ptrs = [_put(data[k][g:g + (b - a)], "device", keep) for (_, _, a, b, g) in mine]
                        fa.fa_accumulate_keys(ctx, k, weights[k], args[0], args[1], ptrs, args[3], s)
                elif op[0] == "final":
                    # read in place: device memory, or pinned memory where the context does
                    # not stage it
                    _, k, key, a, b, g = op
                    kind = "device" if seed % 2 else rng_py.choice(["device", "pinned"])
                    ptr = _put(data[k][g:g + (b - a)], kind, keep)
                    fa.fa_accumulate_final(ctx, k, weights[k], key, a, ptr, b - a, outs, s)
                else:
                    _, k, key, a, b, g = op
                    ptr = _put(data[k][g:g + (b - a)], rng_py.choice(KINDS), keep)
                    fa.fa_accumulate(ctx, k, weights[k], key, a, ptr, b - a, s)
            fa.fa_finalize(ctx, outs, s)
            fa.fa_sync(ctx)
            torch.cuda.synchronize()
            for p, n in enumerate(numels):
                rep = [p in reports[k] for k in range(K)]
                xs = [data[k][offs[p]:offs[p + 1]] for k in range(K)]
                want, N, cnt = oracle.fedavg_key(weights, rep, xs, din, dout)
                assert fa.fa_key_total(ctx, p) == (N, cnt), (rnd, p)
                got = to_np(outs[p], dout)
                what = f"round {rnd} key {p} (n={n}, reporters={cnt})"
                if want is None:
                    assert np.array_equal(got, sentinel_np(n, dout)), what
                    continue
                mx = max(float(np.abs(_as_f32(xs[k], din)).max()) for k in range(K) if rep[k])
                if dout == "f32":
                    check_f32(got, want, mx, cnt, what)
                else:
                    check_f32_to_bf16(got, want, mx, cnt, what)
            del keep
            fa.fa_reset(ctx)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)
