"""The committed ncu summaries describe the kernels as they are: every summary that
records a kernel source digest records the current one, so bench.py's roofline.traffic
(read from them) is never taken from an older kernel."""
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_profile_digests_match_the_kernel_source():
    now = bench.kernel_source_digest()
    seen = 0
    pdir = os.path.join(ROOT, "profiles")
    for name in sorted(os.listdir(pdir)):
        text = open(os.path.join(pdir, name)).read()
        for d in re.findall(r"[Dd]igest[^`]*`([0-9a-f]{16})`", text):
            assert d == now, f"{name} records kernel source {d}, the source is now {now}: retake it"
            seen += 1
    assert seen >= 3


def test_traffic_is_read_for_the_current_source():
    t = bench.profiled_traffic(1288226514)
    assert t is not None and 0.9 * 1288226514 < t < 1.05 * 1288226514
