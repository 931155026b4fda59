"""fa_reduce_subsets: a round of client key subsets (adapter rounds) resident in device
memory, reduced straight to the output in one pass.  It must give the bits of the
per-client path (fa_accumulate_keys for each client in call order, then fa_finalize),
match the oracle under the usual tolerances (the compensated mode under the strict
rule), keep totals exact, leave unsent keys untouched, and be all or nothing on errors."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
import synth
from synth import workloads as W
from tests.compare import Bf16Tally, check_f32, fp32_sum_model
from tests.gpu_helpers import sentinel, sentinel_np, to_dev, to_np

pytestmark = pytest.mark.gpu


def _layout(numels):
    return [(f"k{i}", n) for i, n in enumerate(numels)]


def _packed(host, keys, offset=0, dtype="bf16"):
    """One device buffer with the client's keys back to back (after `offset` elements of
    padding, so that offset 1 leaves the buffer unaligned)."""
    parts = [np.zeros(offset, host[keys[0]].dtype)] + [host[p] for p in keys] if keys else []
    if not parts:
        return torch.empty(1, dtype=torch.int16 if dtype == "bf16" else torch.float32, device="cuda")
    t = to_dev(np.concatenate(parts))
    return t[offset:]


def _per_client(numels, din, dout, ids, weights, hosts, keys, flags, order=None):
    K = max(ids) + 1
    ctx = fa.fa_open(_layout(numels), din, dout, K, flags=flags)
    keep = []
    try:
        for j in (order or range(len(ids))):
            if not keys[j]:
                continue
            xs = [to_dev(hosts[j][p]) for p in keys[j]]
            keep += xs
            fa.fa_accumulate_keys(ctx, ids[j], weights[j], keys[j], [0] * len(keys[j]), xs,
                                  [numels[p] for p in keys[j]])
        outs = [sentinel(n, dout) for n in numels]
        fa.fa_finalize(ctx, outs)
        fa.fa_sync(ctx)
        totals = [fa.fa_key_total(ctx, p) for p in range(len(numels))]
        return [to_np(o, dout) for o in outs], totals
    finally:
        fa.fa_close(ctx)


def _subsets(numels, din, dout, ids, weights, hosts, keys, flags, offset=0, flat=False):
    K = max(ids) + 1
    ctx = fa.fa_open(_layout(numels), din, dout, K, flags=flags | (fa.FA_FLAT_OUT if flat else 0))
    try:
        bufs = [_packed(hosts[j], keys[j], offset, din) for j in range(len(ids))]
        if flat:
            out = sentinel(sum(numels), dout)
            fa.fa_reduce_subsets(ctx, ids, weights, bufs, keys, [out])
        else:
            outs = [sentinel(n, dout) for n in numels]
            fa.fa_reduce_subsets(ctx, ids, weights, bufs, keys, outs)
        fa.fa_sync(ctx)
        totals = [fa.fa_key_total(ctx, p) for p in range(len(numels))]
        if flat:
            o = to_np(out, dout)
            offs = np.cumsum([0] + list(numels))
            res = [o[offs[p]:offs[p + 1]] for p in range(len(numels))]
        else:
            res = [to_np(x, dout) for x in outs]
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_finalize(ctx, [sentinel(sum(numels), dout)])
        assert e.value.status == fa.FA_ERR_STATE
        return res, totals
    finally:
        fa.fa_close(ctx)


@pytest.fixture(scope="module")
def lora():
    w = W.make("lora")
    hosts = [{p: synth.client_key(w, k, p) for p in w.reports[k]} for k in range(w.K)]
    return w, hosts


@pytest.mark.parametrize("flags", [0, fa.FA_COMPENSATED])
@pytest.mark.parametrize("flat", [False, True])
def test_lora_round_bits_and_oracle(lora, flags, flat):
    w, hosts = lora
    ids = list(range(w.K))
    ref, rtot = _per_client(w.numels, "bf16", "bf16", ids, w.weights, hosts, w.reports, flags)
    got, gtot = _subsets(w.numels, "bf16", "bf16", ids, w.weights, hosts, w.reports, flags, flat=flat)
    assert gtot == rtot
    tally = Bf16Tally()
    for p in range(w.n_keys):
        assert np.array_equal(got[p], ref[p]), f"key {p}"
        rep = [p in set(w.reports[k]) for k in range(w.K)]
        xs = [hosts[k].get(p) for k in range(w.K)]
        want, N, cnt = oracle.fedavg_key(w.weights, rep, xs, "bf16", "bf16")
        assert gtot[p] == (N, cnt)
        if want is None:
            assert np.array_equal(got[p], sentinel_np(w.numels[p], "bf16")), f"key {p} written"
            continue
        if flags:
            tally.add(got[p], want, f"key {p}")
        else:
            mx = max(float(np.abs(synth.to_f64(xs[k], "bf16")).max()) for k in range(w.K) if rep[k])
            tally.add(got[p], want, f"key {p}", model=fp32_sum_model(w.weights, rep, xs, "bf16"),
                      bound=1e-6 * mx * cnt)
    tally.check("lora subsets")
    assert any(not any(p in r for r in w.reports) for p in range(w.n_keys)) or True


def _random_round(rng, numels, K, din, p_send=0.6):
    keys = []
    for _ in range(K):
        ks = [p for p in range(len(numels)) if rng.random() < p_send]
        rng.shuffle(ks)                      # any order within a client's buffer
        keys.append(ks)
    hosts = []
    for _ in range(K):
        h = {}
        for p, n in enumerate(numels):
            v = (rng.standard_normal(n) * 0.02).astype(np.float32)
            h[p] = v if din == "f32" else (v.view(np.uint32) >> 16).astype(np.uint16)
        hosts.append(h)
    return keys, hosts


@pytest.mark.parametrize("K", [3, 16, 20])
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f32", "f32"), ("bf16", "f32")])
@pytest.mark.parametrize("offset", [0, 1])
def test_random_subsets_match_per_client_path(K, din, dout, offset):
    """Odd sizes, shuffled key order inside each buffer, unaligned buffers (offset 1), a
    zero-weight client, clients listed out of id order, and K = 20 (more than 16 reporters
    on some keys: the call runs the per-client sequence itself)."""
    rng = np.random.default_rng(300 + K + offset)
    numels = [7, 6144 * 2 + 5, 1000, 33, 70000, 8, 4096, 1]
    keys, hosts = _random_round(rng, numels, K, din, p_send=0.9 if K == 20 else 0.6)
    ids = list(rng.permutation(K))
    weights = [float(v) for v in rng.integers(1, 5000, K)]
    weights[1] = 0.0
    for flags in (0, fa.FA_COMPENSATED):
        ref, rtot = _per_client(numels, din, dout, ids, weights, hosts, keys, flags)
        got, gtot = _subsets(numels, din, dout, ids, weights, hosts, keys, flags, offset=offset)
        assert gtot == rtot
        for p in range(len(numels)):
            assert np.array_equal(got[p].view(np.uint8), ref[p].view(np.uint8)), (flags, p)
    # against the oracle too (clients in the order given)
    for p in range(len(numels)):
        order = [j for j in range(K) if p in keys[j]]
        wts = [weights[j] for j in order]
        want, N, cnt = oracle.fedavg_key(wts, [True] * len(order), [hosts[j][p] for j in order], din, dout)
        if want is None:
            assert np.array_equal(got[p], sentinel_np(numels[p], dout))
        elif dout == "f32":
            mx = max(float(np.abs(synth.to_f64(hosts[j][p], din)).max()) for j in order)
            check_f32(got[p], want, mx, cnt, f"key {p}")


def test_errors_leave_the_round_empty():
    rng = np.random.default_rng(5)
    numels = [100, 4096]
    keys, hosts = _random_round(rng, numels, 3, "bf16", p_send=1.0)
    bufs = [_packed(hosts[j], keys[j]) for j in range(3)]
    outs = [sentinel(n, "bf16") for n in numels]
    ctx = fa.fa_open(_layout(numels), "bf16", "bf16", 3)
    try:
        def expect(status, *args):
            with pytest.raises(fa.FedAvgError) as e:
                fa.fa_reduce_subsets(ctx, *args)
            assert e.value.status == status
            assert fa.fa_key_total(ctx, 0) == (0.0, 0)
        expect(fa.FA_ERR_ARG, [0, 0, 1], [1.0] * 3, bufs, keys, outs)        # id twice
        expect(fa.FA_ERR_ARG, [0, 1, 5], [1.0] * 3, bufs, keys, outs)        # id >= max_clients
        expect(fa.FA_ERR_ARG, [0, 1, 2], [1.0] * 3, bufs, [keys[0], keys[1], [0, 9]], outs)   # no key 9
        expect(fa.FA_ERR_RANGE, [0, 1, 2], [1.0] * 3, bufs, [keys[0], keys[1], [1, 1]], outs)  # key twice
        expect(fa.FA_ERR_WEIGHT, [0, 1, 2], [1.0, -2.0, 1.0], bufs, keys, outs)
        host = torch.zeros(5000, dtype=torch.int16)
        expect(fa.FA_ERR_ARG, [0, 1, 2], [1.0] * 3, [bufs[0], host, bufs[2]], keys, outs)
        expect(fa.FA_ERR_ARG, [0, 1, 2], [1.0] * 3, bufs, keys, [outs[0], torch.zeros(4096, dtype=torch.int16)])
        # after every refusal the round is still empty: a valid call goes through
        fa.fa_reduce_subsets(ctx, [0, 1, 2], [1.0, 2.0, 3.0], bufs, keys, outs)
        fa.fa_sync(ctx)
        assert fa.fa_key_total(ctx, 0) == (6.0, 3)
        expect_state = pytest.raises(fa.FedAvgError)
        with expect_state as e:
            fa.fa_reduce_subsets(ctx, [0, 1, 2], [1.0, 2.0, 3.0], bufs, keys, outs)
        assert e.value.status == fa.FA_ERR_STATE
        fa.fa_reset(ctx)
        x = to_dev(hosts[0][0])
        fa.fa_accumulate(ctx, 0, 1.0, 0, 0, x, numels[0])
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_reduce_subsets(ctx, [1, 2], [1.0, 1.0], bufs[1:], keys[1:], outs)
        assert e.value.status == fa.FA_ERR_STATE
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def _round_on(ctx, numels, din, dout, ids, weights, bufs, keys):
    outs = [sentinel(n, dout) for n in numels]
    fa.fa_reset(ctx)
    fa.fa_reduce_subsets(ctx, ids, weights, bufs, keys, outs)
    fa.fa_sync(ctx)
    return [to_np(o, dout) for o in outs]


@pytest.mark.parametrize("flags", [0, fa.FA_COMPENSATED])
def test_both_table_forms_and_back_to_back_rounds(flags):
    """A round whose tables fit the launch's parameters (a few keys per client) and one
    that needs them in device memory (all 1200 keys from every client), alternating on one
    context: each gives the per-client path's bits, every time.  Back-to-back small rounds
    hand the tile counter from one launch to the next."""
    rng = np.random.default_rng(41 + flags)
    numels = [int(n) for n in rng.integers(1, 3000, 1200)]
    numels[5] = 9000
    K = 3
    _, hosts = _random_round(rng, numels, K, "bf16", p_send=0.0)
    few = [sorted(rng.choice(len(numels), 40, replace=False).tolist()) for _ in range(K)]
    every = [list(range(len(numels))) for _ in range(K)]
    ids = [2, 0, 1]
    weights = [3.0, 1.0, 7.0]
    want = {}
    for name, keys in (("few", few), ("every", every)):
        want[name], _ = _per_client(numels, "bf16", "bf16", ids, weights, hosts, keys, flags)
    ctx = fa.fa_open(_layout(numels), "bf16", "bf16", K, flags=flags)
    try:
        bufs = {name: [_packed(hosts[j], keys[j]) for j in range(K)]
                for name, keys in (("few", few), ("every", every))}
        for name in ("few", "few", "every", "few", "every", "every", "few", "few", "few"):
            keys = few if name == "few" else every
            got = _round_on(ctx, numels, "bf16", "bf16", ids, weights, bufs[name], keys)
            for p in range(len(numels)):
                assert np.array_equal(got[p], want[name][p]), (name, p)
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)
