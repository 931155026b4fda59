"""The device input generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dist", [0, 1])
def test_device_generator_matches_host(dtype, dist):
    for first, n in [(0, 1 << 20), (123456789, 100003), (6_738_415_616 - 5000, 5000)]:
        host = synth.fill(20261206, 3, dist, 0.02, dtype, first, n)
        t = torch.empty(n, dtype=torch.float32 if dtype == "f32" else torch.int16, device="cuda")
        synth.fill_device(20261206, 3, dist, 0.02, dtype, first, n, t.data_ptr(), 0)
        torch.cuda.synchronize()
        got = t.cpu().numpy()
        if dtype == "bf16":
            got = got.view(np.uint16)
        assert np.array_equal(got.view(np.uint8), host.view(np.uint8)), (first, n)
