"""Every element of a full-size bf16 round against the fp64 oracle, key by key.

For each key of the workload the host generator produces every reporting client's
values for that key (in parts, one per host thread), the oracle aggregates them, and
the GPU's output is compared with it under the tolerance of tests/compare.py:
within 1 bf16 ulp everywhere, and >= 99.99 % bit-identical over the whole model.
With `escape` (the default mode), an element may sit more than 1 ulp away only where
the fp32 running sum's own rounding explains it: equal, bit for bit, to fp32_sum_model
and within 1e-6 * max|x| * K + 1 bf16 ulp, max|x| over the key's reporters.  Without
it (the compensated mode) no element may.  Inputs come from the host generator only;
nothing here reads the GPU except the output passed in."""
from __future__ import annotations

import os
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle
import synth
from tests.compare import BF16_MIN_IDENTICAL, bf16_order, bf16_values, fp32_sum_model


class FullTally:
    def __init__(self):
        self.same = 0
        self.total = 0
        self.beyond = 0          # elements > 1 ulp off, each explained by the fp32 sum model
        self.worst = 0           # largest ulp distance seen

    def frac(self) -> float:
        return 1.0 if self.total == 0 else self.same / self.total


def _maxabs_bf16(x: np.ndarray) -> float:
    m = int((x & np.uint16(0x7FFF)).max()) if x.size else 0
    return float(bf16_values(np.array([m], np.uint16))[0])


def compare_every_element(w, got: np.ndarray, escape: bool, threads: int | None = None,
                          part_elems: int = 1 << 22) -> FullTally:
    """got: the flat bf16 output (uint16 bits) of a round in which every client sent every
    key, clients applied in id order.  Raises AssertionError on any element out of
    tolerance; returns the tally."""
    assert w.dtype_in == "bf16" and w.dtype_out == "bf16"
    assert got.dtype == np.uint16 and got.size == w.P
    threads = threads or os.cpu_count() or 1
    rep = [True] * w.K
    tally = FullTally()
    offs = w.flat_offsets()
    t0 = time.time()

    def part(args):
        off, a, b = args
        n = b - a
        xs = [synth.fill(w.seed, k, w.dists[k], w.sigma, "bf16", off + a, n, threads=1)
              for k in range(w.K)]
        want = np.empty(n, np.uint16)
        oracle.fedavg_key(w.weights, rep, xs, "bf16", "bf16", out=want)
        g = got[off + a:off + b]
        d = np.abs(bf16_order(g) - bf16_order(want))
        same = int(np.count_nonzero(d == 0))
        worst = int(d.max()) if d.size else 0
        over = np.flatnonzero(d > 1)
        esc = None
        if over.size:
            assert escape, f"{n} elements at flat {off + a}: {over.size} beyond 1 ulp (worst {worst})"
            model = fp32_sum_model(w.weights, rep, [x[over] for x in xs], "bf16")
            assert np.array_equal(g[over], model), \
                f"flat {off + a}: {over.size} elements beyond 1 ulp that the fp32 sum does not explain"
            esc = (g[over].copy(), want[over].copy())
        part_max = max(_maxabs_bf16(x) for x in xs) if escape else 0.0
        return same, n, worst, esc, part_max

    with ThreadPoolExecutor(threads) as ex:
        # every part of every key queued at once, so that all threads stay busy
        futs = []
        for p in range(w.n_keys):
            off, n = offs[p], w.numels[p]
            cuts = list(range(0, n, part_elems)) + [n]
            futs.append([ex.submit(part, (off, a, b)) for a, b in zip(cuts[:-1], cuts[1:])])
        for p, fs in enumerate(futs):
            key_max = 0.0
            escaped = []
            for f in fs:
                same, tot, worst, esc, part_max = f.result()
                tally.same += same
                tally.total += tot
                tally.worst = max(tally.worst, worst)
                key_max = max(key_max, part_max)
                if esc is not None:
                    escaped.append(esc)
            # escaped elements stay within the fp32 bound, max|x| over the key's reporters
            for gb, wb in escaped:
                gv, wv = bf16_values(gb), bf16_values(wb)
                ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(wv), 2.0 ** -126))) - 7)
                assert (np.abs(gv - wv) <= 1e-6 * key_max * w.K + ulp).all(), f"key {p}: beyond the fp32 bound"
                tally.beyond += gb.size
    assert tally.total == w.P
    assert tally.frac() >= BF16_MIN_IDENTICAL, f"only {tally.frac():.6%} bit-identical"
    print(f"{w.name}: every element ({tally.total}) compared in {time.time() - t0:.0f} s on "
          f"{threads} threads: {tally.frac():.6%} bit-identical, {tally.beyond} beyond 1 ulp "
          f"(each equal to the fp32 sum model), worst {tally.worst} ulp")
    return tally
