"""Host bookkeeping of a round (CPU, via the host-only ledger shim): argument
validation, flat chunks split at key boundaries, which elements take their
first contribution, per-client element counts, per-key weight totals N_p and
reporter counts (bit-exact against the oracle's totals), round state."""
import random

import numpy as np
import pytest

import oracle
from tests.ledger import Ledger

OK, ARG, RANGE, WEIGHT, INCOMPLETE, STATE = 0, -1, -2, -4, -5, -6


def test_padding_is_32_elements():
    lg = Ledger([1, 33, 64, 7], 2)
    assert [lg.acc_off(p) for p in range(4)] == [0, 32, 96, 160]
    assert lg.padded() == 192


def test_bad_layouts():
    assert Ledger([], 1).status == ARG
    assert Ledger([3, 0], 1).status == ARG
    assert Ledger([3], 0).status == ARG


def test_weight_validation():
    lg = Ledger([10], 3)
    for w in (-1.0, float("nan"), float("inf"), 2.0 ** 24 + 1):
        assert lg.accumulate([0], [w], 0, 0, 5)[0] == WEIGHT
    assert lg.accumulate([0], [2.0 ** 24], 0, 0, 5)[0] == OK
    assert lg.accumulate([0], [7.0], 0, 5, 5)[0] == WEIGHT        # unlike its first chunk
    assert lg.accumulate([0], [2.0 ** 24], 0, 5, 5)[0] == OK
    assert lg.accumulate([1], [0.0], 0, 0, 10)[0] == OK           # zero weight is allowed


def test_empty_chunk_registers_nothing():
    lg = Ledger([10], 2)
    assert lg.accumulate([0], [5.0], 0, 3, 0) == (OK, [])
    assert lg.accumulate([0], [6.0], 0, 0, 10)[0] == OK           # weight not fixed by the empty call
    assert lg.key_total(0) == (OK, 6.0, 1)


def test_ids_keys_ranges():
    lg = Ledger([10, 20], 2)
    assert lg.accumulate([2], [1.0], 0, 0, 1)[0] == ARG
    assert lg.accumulate([0, 0], [1.0, 1.0], 0, 0, 1)[0] == ARG
    assert lg.accumulate([0], [1.0], 2, 0, 1)[0] == ARG
    assert lg.accumulate([0], [1.0], -2, 0, 1)[0] == ARG
    assert lg.accumulate([0], [1.0], 0, 0, 11)[0] == RANGE
    assert lg.accumulate([0], [1.0], 0, 11, 0)[0] == RANGE
    assert lg.accumulate([0], [1.0], 0, 2 ** 64 - 1, 2)[0] == RANGE   # no wrap-around
    assert lg.accumulate([0], [1.0], -1, 25, 6)[0] == RANGE
    assert lg.accumulate([0], [1.0], -1, 25, 5)[0] == OK


def test_flat_chunk_splits_at_keys():
    lg = Ledger([10, 20, 5], 1)
    st, pieces = lg.accumulate([0], [1.0], -1, 8, 24)
    assert st == OK
    # (key, chunk_off, acc_idx, len, first)
    assert pieces == [(0, 0, 8, 2, 1), (1, 2, 32, 20, 1), (2, 22, 64, 2, 1)]


def test_first_contribution_tracking():
    lg = Ledger([5, 20], 2)
    assert lg.accumulate([0], [1.0], 1, 0, 10)[1] == [(1, 0, 32, 10, 1)]
    assert lg.accumulate([1], [1.0], 1, 5, 10)[1] == [(1, 0, 37, 5, 0), (1, 5, 42, 5, 1)]
    assert lg.accumulate([0], [1.0], 1, 10, 10)[1] == [(1, 0, 42, 5, 0), (1, 5, 47, 5, 1)]
    assert lg.accumulate([1], [1.0], 1, 0, 5)[1] == [(1, 0, 32, 5, 0)]
    assert lg.accumulate([1], [1.0], 1, 15, 5)[1] == [(1, 0, 47, 5, 0)]


def test_over_coverage_and_incomplete():
    lg = Ledger([10], 2)
    assert lg.accumulate([0], [1.0], 0, 0, 6)[0] == OK
    assert lg.accumulate([0], [1.0], 0, 0, 5)[0] == RANGE         # 6 + 5 > 10
    st, items = lg.finalize()
    assert st == INCOMPLETE
    assert lg.accumulate([0], [1.0], 0, 6, 4)[0] == OK
    st, items = lg.finalize()
    assert st == OK and items == [(0, 0, 0, 10, 1, 1.0)]


def test_finalize_skips_unsent_and_zero_weight_keys_then_closes():
    lg = Ledger([4, 4, 4], 3)
    lg.accumulate([0], [0.0], 1, 0, 4)
    lg.accumulate([1], [0.0], 1, 0, 4)
    lg.accumulate([2], [3.0], 2, 0, 4)
    st, items = lg.finalize()
    assert st == OK
    assert items == [(2, 64, 8, 4, 1, 3.0)]
    assert lg.key_total(1) == (OK, 0.0, 2)
    assert lg.accumulate([2], [3.0], 0, 0, 1)[0] == STATE
    lg.reset()
    assert lg.key_total(2) == (OK, 0.0, 0)
    assert lg.accumulate([2], [9.0], 0, 0, 4)[1] == [(0, 0, 0, 4, 1)]


def test_batch_starts_sum_once():
    lg = Ledger([8, 8], 4)
    st, pieces = lg.accumulate([3, 1, 2], [1.0, 2.0, 3.0], -1, 4, 8)
    assert st == OK and pieces == [(0, 0, 4, 4, 1), (1, 4, 32, 4, 1)]
    assert lg.key_total(0) == (OK, 6.0, 3)


def test_totals_bit_exact_with_oracle():
    """Random partial participation: N_p and |S_p| equal the oracle's, bit for bit."""
    rng = np.random.default_rng(5)
    numels = [int(v) for v in rng.integers(1, 50, 30)]
    K = 9
    weights = [float(v) for v in rng.integers(0, 5000, K)] 
    weights[3] = 0.1            # non-integer weights sum in client order too
    weights[5] = 1e-3
    lg = Ledger(numels, K)
    reports = [[p for p in range(len(numels)) if rng.random() < 0.6] for _ in range(K)]
    order = [(k, p) for k in range(K) for p in reports[k]]
    random.Random(1).shuffle(order)
    for k, p in order:
        assert lg.accumulate([k], [weights[k]], p, 0, numels[p])[0] == OK
    st, items = lg.finalize()
    assert st == OK
    by_key = {it[0]: it for it in items}
    for p, n in enumerate(numels):
        rep = [p in reports[k] for k in range(K)]
        xs = [np.zeros(n, np.float32)] * K
        _, N, cnt = oracle.fedavg_key(weights, rep, xs, "f32", "f32")
        assert lg.key_total(p) == (OK, N, cnt)
        if cnt and N > 0:
            assert by_key[p][4] == cnt and by_key[p][5] == N
        else:
            assert p not in by_key


def test_random_operations_against_model():
    """Random chunked traffic against a plain per-element model of the bookkeeping."""
    rng = random.Random(11)
    for trial in range(30):
        numels = [rng.randint(1, 40) for _ in range(rng.randint(1, 6))]
        K = rng.randint(1, 5)
        lg = Ledger(numels, K)
        offs = np.cumsum([0] + numels)
        started = [np.zeros(n, bool) for n in numels]
        recv = np.zeros((K, len(numels)), np.int64)
        weight = {}
        for _ in range(60):
            J = rng.randint(1, K)
            clients = rng.sample(range(K), J)
            ws = [weight.get(c, float(rng.randint(0, 9))) for c in clients]
            if rng.random() < 0.5:
                key = -1
                off = rng.randint(0, int(offs[-1]))
                ln = rng.randint(0, int(offs[-1]) - off)
            else:
                key = rng.randrange(len(numels))
                off = rng.randint(0, numels[key])
                ln = rng.randint(0, numels[key] - off)
            # expected status
            spans = []
            if key == -1:
                pos = off
                while pos < off + ln:
                    p = int(np.searchsorted(offs, pos, side="right") - 1)
                    e = min(off + ln, int(offs[p + 1]))
                    spans.append((p, pos - int(offs[p]), e - pos, pos - off))
                    pos = e
            elif ln:
                spans.append((key, off, ln, 0))
            over = any(recv[c, p] + n > numels[p] for c in clients for (p, _, n, _) in spans)
            st, pieces = lg.accumulate(clients, ws, key, off, ln)
            if over:
                assert st == RANGE
                continue
            assert st == OK
            if ln == 0:
                assert pieces == []
                continue
            for c, w in zip(clients, ws):
                weight[c] = w
                for (p, _, n, _) in spans:
                    recv[c, p] += n
            # element-wise first flags
            got = {}
            for (p, coff, acc, n, first) in pieces:
                for i in range(n):
                    got[(p, acc - lg.acc_off(p) + i)] = (first, coff + i)
            for (p, koff, n, coff) in spans:
                for i in range(n):
                    f, ci = got.pop((p, koff + i))
                    assert ci == coff + i
                    assert f == (0 if started[p][koff + i] else 1)
                    started[p][koff + i] = True
            assert not got
        for p in range(len(numels)):
            rep = [k for k in range(K) if recv[k, p] > 0]
            assert lg.key_total(p) == (OK, sum(weight[k] for k in rep), len(rep))
        st, items = lg.finalize()
        complete = all(recv[k, p] in (0, numels[p]) for k in range(K) for p in range(len(numels)))
        assert st == (OK if complete else INCOMPLETE)


def _spans(numels, offs, key, off, ln):
    spans = []
    if key == -1:
        pos = off
        while pos < off + ln:
            p = int(np.searchsorted(offs, pos, side="right") - 1)
            e = min(off + ln, int(offs[p + 1]))
            spans.append((p, pos - int(offs[p]), e - pos, pos - off))
            pos = e
    elif ln:
        spans.append((key, off, ln, 0))
    return spans


def test_accumulate_keys_against_model():
    """One client's several chunks per call: the same pieces, first-contribution flags and
    counts as the chunks sent one by one would give; over-coverage is seen across chunks
    of the call; on any error nothing is recorded."""
    rng = random.Random(23)
    for trial in range(40):
        numels = [rng.randint(1, 30) for _ in range(rng.randint(1, 6))]
        K = rng.randint(1, 4)
        lg = Ledger(numels, K)
        offs = np.cumsum([0] + numels)
        started = [np.zeros(n, bool) for n in numels]
        recv = np.zeros((K, len(numels)), np.int64)
        weight = {}
        for _ in range(40):
            c = rng.randrange(K)
            w = weight.get(c, float(rng.randint(0, 9)))
            chunks = []
            for _ in range(rng.randint(0, 5)):
                if rng.random() < 0.3:
                    off = rng.randint(0, int(offs[-1]))
                    chunks.append((-1, off, rng.randint(0, int(offs[-1]) - off)))
                else:
                    key = rng.randrange(len(numels))
                    off = rng.randint(0, numels[key])
                    chunks.append((key, off, rng.randint(0, numels[key] - off)))
            if rng.random() < 0.1 and chunks:                 # a chunk past the end
                i = rng.randrange(len(chunks))
                k, o, n = chunks[i]
                chunks[i] = (k, o, (offs[-1] if k == -1 else numels[k]) - o + 1)
                bad_range = True
            else:
                bad_range = False
            before = [lg.key_total(p) for p in range(len(numels))]
            st, pieces = lg.accumulate_keys(c, w, chunks)
            pending = recv[c].copy()
            over = False
            for (k, o, n) in ([] if bad_range else chunks):
                for (p, _, m, _) in _spans(numels, offs, k, o, n):
                    pending[p] += m
                    over = over or pending[p] > numels[p]
            if bad_range or over:
                assert st == RANGE, (st, lg.error())
                assert pieces == []
                assert [lg.key_total(p) for p in range(len(numels))] == before
                continue
            assert st == OK, lg.error()
            if all(n == 0 for (_, _, n) in chunks):
                assert pieces == []
                continue
            weight[c] = w
            recv[c] = pending
            got = {}
            for (ch, p, coff, acc, n, first) in pieces:
                for i in range(n):
                    got[(ch, p, acc - lg.acc_off(p) + i)] = (first, coff + i)
            for ch, (k, o, n) in enumerate(chunks):
                for (p, koff, m, coff) in _spans(numels, offs, k, o, n):
                    for i in range(m):
                        f, ci = got.pop((ch, p, koff + i))
                        assert ci == coff + i
                        assert f == (0 if started[p][koff + i] else 1)
                        started[p][koff + i] = True
            assert not got
        for p in range(len(numels)):
            rep = [k for k in range(K) if recv[k, p] > 0]
            assert lg.key_total(p) == (OK, sum(weight[k] for k in rep), len(rep))


def test_accumulate_keys_errors_record_nothing():
    lg = Ledger([10, 20], 2)
    assert lg.accumulate_keys(0, 5.0, [(0, 0, 10), (1, 0, 20)])[0] == OK
    # weight unlike the client's earlier chunks, bad key, bad client: nothing recorded
    assert lg.accumulate_keys(0, 6.0, [(0, 0, 1)])[0] == WEIGHT
    assert lg.accumulate_keys(1, 3.0, [(0, 0, 10), (7, 0, 1)])[0] == ARG
    assert "chunk 1" in lg.error()
    assert lg.accumulate_keys(2, 3.0, [(0, 0, 10)])[0] == ARG
    # two chunks of one key in one call that together exceed it
    assert lg.accumulate_keys(1, 3.0, [(1, 0, 15), (1, 0, 15)])[0] == RANGE
    assert lg.key_total(0) == (OK, 5.0, 1) and lg.key_total(1) == (OK, 5.0, 1)
    # client 1 can still send everything
    st, pieces = lg.accumulate_keys(1, 3.0, [(-1, 0, 30)])
    assert st == OK and [p[0] for p in pieces] == [0, 0]
    assert lg.key_total(1) == (OK, 8.0, 2)
    assert lg.finalize()[0] == OK
    assert lg.accumulate_keys(1, 3.0, [(0, 0, 1)])[0] == STATE


def test_accumulate_keys_matches_single_calls():
    """The pieces of a multi-chunk call equal those of the same chunks sent one by one."""
    numels = [7, 33, 1, 64, 5]
    a, b = Ledger(numels, 3), Ledger(numels, 3)
    calls = [(0, 2.0, [(1, 0, 10), (3, 5, 20), (-1, 0, 7)]),
             (1, 4.0, [(-1, 3, 50), (4, 0, 5)]),
             (0, 2.0, [(1, 10, 23), (3, 0, 5), (3, 25, 39), (2, 0, 1)])]
    for c, w, chunks in calls:
        st, multi = a.accumulate_keys(c, w, chunks)
        assert st == OK, a.error()
        single = []
        for (k, o, n) in chunks:
            st, ps = b.accumulate([c], [w], k, o, n)
            assert st == OK, b.error()
            single += [tuple(int(v) for v in q) for q in ps]
        assert [tuple(int(v) for v in q[1:]) for q in multi] == single
    assert [a.key_total(p) for p in range(5)] == [b.key_total(p) for p in range(5)]


def test_whole_keys_records_like_accumulate_keys():
    """record_whole_keys (the round-level subset reduce's bookkeeping) leaves the same totals,
    reporter counts and finalize list as accumulate_keys with whole keys."""
    numels = [5, 100, 7, 64, 1]
    rng = random.Random(11)
    for trial in range(20):
        K = rng.randint(1, 6)
        a, b = Ledger(numels, K + 2), Ledger(numels, K + 2)
        for c in rng.sample(range(K + 2), K):
            keys = rng.sample(range(len(numels)), rng.randint(0, len(numels)))
            w = float(rng.choice([0, 1, 3, 1000, 2 ** 24]))
            assert a.whole_keys(c, w, keys) == 0
            st, _ = b.accumulate_keys(c, w, [(p, 0, numels[p]) for p in keys])
            assert st == 0
        for p in range(len(numels)):
            assert a.key_total(p) == b.key_total(p)
        assert a.finalize() == b.finalize()


def test_whole_keys_errors_record_nothing():
    numels = [5, 100, 7]
    lg = Ledger(numels, 3)
    assert lg.whole_keys(0, 2.0, [0, 2]) == 0
    before = [lg.key_total(p) for p in range(3)]
    assert lg.whole_keys(1, 1.0, [1, 3]) == -1          # key out of range
    assert lg.whole_keys(1, 1.0, [1, -1]) == -1         # flat is not a whole key
    assert lg.whole_keys(1, 1.0, [1, 2, 1]) == -2       # the same key twice
    assert lg.whole_keys(0, 2.0, [1, 0]) == -2          # key 0 already sent by client 0
    assert lg.whole_keys(0, 3.0, [1]) == -4             # weight differs from earlier
    assert lg.whole_keys(2, -1.0, [1]) == -4            # invalid weight
    assert lg.whole_keys(5, 1.0, [1]) == -1             # client id out of range
    assert [lg.key_total(p) for p in range(3)] == before
    assert lg.whole_keys(1, 1.0, [1, 2]) == 0           # still accepted afterwards
    assert lg.key_total(2) == (0, 3.0, 2)
    st, _ = lg.finalize()
    assert st == 0
    assert lg.whole_keys(2, 1.0, [0]) == -6             # closed


# ------------------------------------------------------------------ final contributions
# fa_accumulate_final: the last contribution to a range, fused with its finalize.  N_p is
# final once every other sender of the key has sent all of it; the key then takes no new
# sender, the range no further contribution, and fa_finalize writes only the rest.

def test_final_contribution_totals_and_written_ranges():
    lg = Ledger([10, 6], 3)
    assert lg.accumulate([0], [2.0], 0, 0, 10)[0] == OK
    assert not lg.has_final()
    st, pieces, totals = lg.accumulate_final(1, 3.0, 0, 0, 4)
    assert st == OK and pieces == [(0, 0, 0, 4, 0)] and totals == [5.0]
    assert lg.has_final()
    # the rest of key 0 through a plain call, key 1 untouched by any final call
    assert lg.accumulate([1], [3.0], 0, 4, 6)[0] == OK
    assert lg.accumulate([2], [1.0], 1, 0, 6)[0] == OK
    st, items = lg.finalize_ranges()
    assert st == OK
    assert items == [(0, 4, 4, 4, 6, 2, 5.0), (1, 0, 32, 10, 6, 1, 1.0)]
    # everything written by final calls: nothing left for fa_finalize
    lg.reset()
    assert not lg.has_final()
    lg.accumulate([0], [2.0], 0, 0, 10)
    st, _, totals = lg.accumulate_final(1, 3.0, 0, 0, 10)
    assert st == OK and totals == [5.0]
    assert lg.finalize_ranges() == (OK, [])


def test_final_needs_every_other_sender_complete():
    lg = Ledger([10], 3)
    assert lg.accumulate([0], [2.0], 0, 0, 6)[0] == OK
    st, pieces, _ = lg.accumulate_final(1, 3.0, 0, 0, 10)
    assert st == INCOMPLETE and pieces == []
    assert lg.key_total(0) == (OK, 2.0, 1)               # nothing recorded
    assert not lg.has_final()
    assert lg.accumulate([1], [3.0], 0, 0, 10)[0] == OK  # the key is not frozen
    assert lg.accumulate([0], [2.0], 0, 6, 4)[0] == OK
    assert lg.finalize_ranges()[1] == [(0, 0, 0, 0, 10, 2, 5.0)]


def test_frozen_key_refuses_new_senders_and_written_ranges():
    lg = Ledger([8, 8], 4)
    lg.accumulate([0], [1.0], 0, 0, 8)
    assert lg.accumulate_final(1, 2.0, 0, 2, 3)[0] == OK            # [2, 5) written
    assert lg.accumulate([2], [4.0], 0, 0, 8)[0] == STATE            # new sender of a frozen key
    assert lg.accumulate_keys(2, 4.0, [(0, 0, 1)])[0] == STATE
    assert lg.whole_keys(2, 4.0, [0]) == STATE
    assert lg.accumulate([1], [2.0], 0, 4, 2)[0] == STATE            # overlaps [2, 5)
    assert lg.accumulate_final(1, 2.0, 0, 0, 3)[0] == STATE
    # all or nothing: a keys call with one bad chunk records none of them
    assert lg.accumulate_keys(1, 2.0, [(0, 0, 2), (0, 4, 1)])[0] == STATE
    assert lg.key_total(0) == (OK, 3.0, 2)
    assert lg.accumulate([1], [2.0], 0, 0, 2)[0] == OK               # outside the written range
    assert lg.accumulate_final(1, 2.0, 0, 5, 3)[0] == OK
    assert lg.accumulate([2], [4.0], 1, 0, 8)[0] == OK               # key 1 is not frozen
    st, items = lg.finalize_ranges()
    assert st == OK and items == [(0, 0, 0, 0, 2, 2, 3.0), (1, 0, 32, 8, 8, 1, 4.0)]
    lg.reset()                                                        # a new round forgets it all
    assert lg.accumulate([2], [4.0], 0, 0, 8)[0] == OK


def test_final_flat_chunk_across_keys_and_sole_sender():
    lg = Ledger([5, 7, 3], 2)
    lg.accumulate([0], [2.0], 1, 0, 7)
    # client 1: a flat chunk over the end of key 0, all of key 1, the start of key 2;
    # keys 0 and 2 have no other sender (first contribution, N_p = 6), key 1 has client 0
    st, pieces, totals = lg.accumulate_final(1, 6.0, -1, 3, 10)
    assert st == OK
    assert pieces == [(0, 0, 3, 2, 1), (1, 2, 32, 7, 0), (2, 9, 64, 1, 1)]
    assert totals == [6.0, 8.0, 6.0]
    st, items = lg.finalize_ranges()
    assert st == INCOMPLETE                                           # client 1 owes the rest of keys 0, 2
    assert lg.accumulate([1], [6.0], -1, 0, 3)[0] == OK
    assert lg.accumulate([1], [6.0], 2, 1, 2)[0] == OK
    st, items = lg.finalize_ranges()
    assert st == OK and items == [(0, 0, 0, 0, 3, 1, 6.0), (2, 1, 65, 13, 2, 1, 6.0)]


def test_final_zero_weight_key_reports_a_zero_total():
    lg = Ledger([4], 2)
    lg.accumulate([0], [0.0], 0, 0, 4)
    st, _, totals = lg.accumulate_final(1, 0.0, 0, 0, 4)
    assert st == OK and totals == [0.0]
    assert lg.finalize_ranges() == (OK, [])


def test_random_final_contributions_against_model():
    """Random plain and final contributions (per key and flat) against a per-element model
    of the rules: a final chunk needs every other sender of its keys complete, then those
    keys take no new sender and its range no further contribution; totals count every
    sender; finalize writes each key less the ranges final chunks wrote."""
    rng = random.Random(23)
    for trial in range(40):
        numels = [rng.randint(1, 24) for _ in range(rng.randint(1, 5))]
        K = rng.randint(2, 5)
        lg = Ledger(numels, K)
        offs = np.cumsum([0] + numels)
        nk = len(numels)
        started = [np.zeros(n, bool) for n in numels]
        written = [np.zeros(n, bool) for n in numels]
        frozen = [False] * nk
        recv = np.zeros((K, nk), np.int64)
        weight = {}
        for _ in range(50):
            c = rng.randrange(K)
            w = weight.get(c, float(rng.randint(0, 9)))
            if rng.random() < 0.4:
                key = -1
                off = rng.randint(0, int(offs[-1]))
                ln = rng.randint(0, int(offs[-1]) - off)
            else:
                key = rng.randrange(nk)
                off = rng.randint(0, numels[key])
                ln = rng.randint(0, numels[key] - off)
            final = rng.random() < 0.3
            spans = _spans(numels, offs, key, off, ln)
            want = OK
            for (p, koff, n, _) in spans:
                if recv[c, p] + n > numels[p]:
                    want = RANGE
                    break
                if final and any(0 < recv[o, p] < numels[p] for o in range(K) if o != c):
                    want = INCOMPLETE
                    break
            if want == OK:
                for (p, koff, n, _) in spans:
                    if frozen[p] and (recv[c, p] == 0 or written[p][koff:koff + n].any()):
                        want = STATE
                        break
            if final:
                st, pieces, totals = lg.accumulate_final(c, w, key, off, ln)
            else:
                st, pieces = lg.accumulate([c], [w], key, off, ln)
            assert st == want, (trial, final, key, off, ln, st, want)
            if st != OK or ln == 0:
                assert pieces == []
                continue
            weight[c] = w
            for (p, _, n, _) in spans:
                recv[c, p] += n
            got = {}
            for (p, coff, acc, n, first) in pieces:
                for i in range(n):
                    got[(p, acc - lg.acc_off(p) + i)] = (first, coff + i)
            for (p, koff, n, coff) in spans:
                for i in range(n):
                    f, ci = got.pop((p, koff + i))
                    assert ci == coff + i
                    assert f == (0 if started[p][koff + i] else 1)
                    started[p][koff + i] = True
            assert not got
            if final:
                for (p, koff, n, _) in spans:
                    frozen[p] = True
                    written[p][koff:koff + n] = True
                for (p, _, _, _, _), tot in zip(pieces, totals):
                    assert tot == sum(weight[k] for k in range(K) if recv[k, p] > 0)
        assert lg.has_final() == any(wr.any() for wr in written)
        st, items = lg.finalize_ranges()
        complete = all(recv[k, p] in (0, numels[p]) for k in range(K) for p in range(nk))
        assert st == (OK if complete else INCOMPLETE)
        if not complete:
            continue
        want_items = []
        for p in range(nk):
            rep = [k for k in range(K) if recv[k, p] > 0]
            total = sum(weight[k] for k in rep)
            if not rep or total == 0.0:
                continue
            a = 0
            while a < numels[p]:
                if written[p][a]:
                    a += 1
                    continue
                b = a
                while b < numels[p] and not written[p][b]:
                    b += 1
                want_items.append((p, a, lg.acc_off(p) + a, int(offs[p]) + a, b - a, len(rep), total))
                a = b
        assert items == want_items, trial
