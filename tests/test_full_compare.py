"""The every-element comparison used by the full-size GPU parity tests, checked on the
CPU: an output equal to the oracle passes at 100 %, a 1-ulp change passes but is
counted, a 2-ulp change fails (with or without the fp32-sum escape, since it does not
equal the fp32 sum model), and so does a key left unwritten."""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads as W
from tests.compare import bf16_order
from tests.full_compare import compare_every_element


def _workload():
    keys = [("a", (1000,)), ("b", (700, 100)), ("c", (3,)), ("d", (4097,))]
    K = 5
    dists = [W.DIST_NORMAL] * K
    dists[3] = W.DIST_STUDENT3
    w = W.Workload("small", 99, keys, K, "bf16", "bf16", 0.02, [300.0, 17.0, 4096.0, 1.0, 999.0],
                   [list(range(len(keys)))] * K, dists, 0, 12345)
    return W._finish(w)


def _oracle_output(w):
    xs = [synth.client_flat(w, k, 0, w.P) for k in range(w.K)]
    out, _, _ = oracle.fedavg_key(w.weights, [True] * w.K, xs, "bf16", "bf16")
    return out


def _step(bits, ulps):
    """Move bf16 values by `ulps` in value order (away from zero for positive steps)."""
    o = bf16_order(bits) + ulps
    mag = np.abs(o).astype(np.uint16)
    return np.where(o < 0, mag | np.uint16(0x8000), mag).astype(np.uint16)


@pytest.mark.parametrize("escape", [False, True])
def test_exact_output_passes(escape):
    w = _workload()
    t = compare_every_element(w, _oracle_output(w), escape, threads=3, part_elems=997)
    assert t.total == w.P and t.same == w.P and t.beyond == 0


def test_one_ulp_is_counted_two_ulps_fail():
    w = _workload()
    good = _oracle_output(w)
    got = good.copy()
    got[[5, 1500, w.P - 1]] = _step(got[[5, 1500, w.P - 1]], 1)
    t = compare_every_element(w, got, False, threads=2, part_elems=1 << 10)
    assert t.same == w.P - 3 and t.worst == 1
    got[7000] = _step(got[7000:7001], 2)[0]
    for escape in (False, True):
        with pytest.raises(AssertionError):
            compare_every_element(w, got, escape, threads=2, part_elems=1 << 10)


def test_unwritten_key_fails():
    w = _workload()
    got = _oracle_output(w)
    off = w.flat_offsets()[3]
    got[off:off + w.numels[3]] = 0x7FBF
    with pytest.raises(AssertionError):
        compare_every_element(w, got, True, threads=2)
