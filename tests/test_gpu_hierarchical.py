"""Hierarchical FedAvg on the GPU: clients grouped into silos, each silo averaged
by its own context (fp32 output), then the silo means averaged by a top-level
context with each silo's weight total as its weight -- the HFL-DDP regime of
"Technical Summary: Adaptive Data Partitioning for Energy-Efficient Federated and
Distributed Learning in Heterogeneous Systems" (section 2, "Execution regimes",
item 3).  The result must match the flat weighted mean over all clients (the
oracle) within tolerance: the silo means' fp32 rounding is the only extra error."""
import numpy as np
import pytest
import torch

import oracle
import server_side_fedavg_gb300 as fa
from tests.compare import check_f32, check_f32_to_bf16
from tests.gpu_helpers import to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_two_level_matches_flat_oracle(dout):
    rng = np.random.default_rng(51)
    numels = [4097, 30000, 7, 65536]
    layout = [(f"k{i}", n) for i, n in enumerate(numels)]
    K = 11
    w = [float(v) for v in rng.integers(50, 5000, K)]
    xs = [[((rng.standard_normal(n) * 0.02).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
           for n in numels] for _ in range(K)]
    silos = [[0, 1, 2], [3, 4, 5, 6], [7], [8, 9, 10]]
    means, totals = [], []
    for members in silos:
        ctx = fa.fa_open(layout, "bf16", "f32", len(members))
        try:
            for j, k in enumerate(members):
                for p, n in enumerate(numels):
                    fa.fa_accumulate(ctx, j, w[k], p, 0, to_dev(xs[k][p]), n)
            outs = [torch.empty(n, dtype=torch.float32, device="cuda") for n in numels]
            fa.fa_finalize(ctx, outs)
            means.append(outs)
            totals.append(fa.fa_key_total(ctx, 0)[0])
        finally:
            fa.fa_close(ctx)
    top = fa.fa_open(layout, "f32", dout, len(silos))
    try:
        for s, outs in enumerate(means):
            for p, n in enumerate(numels):
                fa.fa_accumulate(top, s, totals[s], p, 0, outs[p], n)
        res = [torch.empty(n, dtype=torch.float32 if dout == "f32" else torch.int16, device="cuda")
               for n in numels]
        fa.fa_finalize(top, res)
        torch.cuda.synchronize()
        assert fa.fa_key_total(top, 0) == (sum(w), len(silos))
    finally:
        fa.fa_close(top)
    for p, n in enumerate(numels):
        want, N, cnt = oracle.fedavg_key(w, [True] * K, [xs[k][p] for k in range(K)], "bf16", dout)
        got = to_np(res[p], dout)
        mx = max(float(np.abs((xs[k][p].astype(np.uint32) << 16).view(np.float32)).max()) for k in range(K))
        if dout == "f32":
            check_f32(got, want, mx, K, f"key {p}")
        else:
            # the top level's inputs are fp32 silo means: its products round in the fp32
            # sum, so the fp32-input rule applies (fp32 bound plus one bf16 ulp)
            check_f32_to_bf16(got, want, mx, K, f"key {p}")
