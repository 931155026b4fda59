"""The committed ncu figures describe the kernels as they are: every machine-readable
profile summary (profiles/*.json) records the digest of the sources its kernel is built
from, and that digest matches those files now, so bench.py's roofline.traffic (read from
one of them) is never taken from an older kernel."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _summaries():
    pdir = os.path.join(ROOT, "profiles")
    return {n: json.load(open(os.path.join(pdir, n))) for n in sorted(os.listdir(pdir))
            if n.endswith(".json")}


def test_profile_digests_match_the_kernel_source():
    sums = _summaries()
    assert len(sums) >= 5, sorted(sums)
    for name, d in sums.items():
        srcs = d["sources"]
        assert srcs and all(any(s in fs for fs in bench.KERNEL_SOURCES.values()) for s in srcs), name
        now = bench.kernel_source_digest(srcs)
        assert d["kernel_source_digest"] == now, \
            f"{name} records kernel source {d['kernel_source_digest']}, the source is now {now}: retake it"
        assert d["command"].startswith("ncu ") and "--clock-control none" in d["command"], name


def test_traffic_is_read_for_the_current_source():
    t = bench.profiled_traffic(1288226514)
    assert t is not None and 0.9 * 1288226514 < t < 1.05 * 1288226514
