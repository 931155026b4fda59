"""Host input generator: determinism, counter access, distribution shape, and
the workload tables (sizes from the configurations' stated shapes)."""
import numpy as np
import pytest

import synth
from synth import workloads as W


def test_counter_access_matches_fill():
    a = synth.fill(123, 3, 0, 0.05, "f32", 1000, 5000)
    idx = np.arange(1000, 6000, dtype=np.uint64)
    b = synth.gather(123, 3, 0, 0.05, "f32", idx)
    assert np.array_equal(a, b)
    c = synth.fill(123, 3, 0, 0.05, "f32", 3000, 10)
    assert np.array_equal(c, a[2000:2010])


def test_threaded_fill_is_deterministic():
    a = synth.fill(5, 0, 0, 0.02, "bf16", 0, 1 << 20, threads=1)
    b = synth.fill(5, 0, 0, 0.02, "bf16", 0, 1 << 20, threads=7)
    assert np.array_equal(a, b)


def test_bf16_is_truncated_f32():
    f = synth.fill(9, 1, 0, 0.02, "f32", 0, 10000)
    h = synth.fill(9, 1, 0, 0.02, "bf16", 0, 10000)
    assert np.array_equal((f.view(np.uint32) >> 16).astype(np.uint16), h)


def test_normal_moments():
    x = synth.fill(1, 0, 0, 1.0, "f32", 0, 1 << 21).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert np.abs(x).max() <= 6.0
    k = ((x - x.mean()) ** 4).mean() / x.var() ** 2 - 3.0
    assert abs(k - (-0.1)) < 0.03          # Irwin-Hall(12) excess kurtosis is -1/10


def test_student_t_heavy_tails():
    x = synth.fill(2, 0, 1, 1.0, "f32", 0, 1 << 19).astype(np.float64)
    assert abs(np.median(x)) < 0.01
    # Student-t(3): P(|t| > 5) ~ 1.54%; a normal would give ~6e-7
    assert 0.01 < np.mean(np.abs(x) > 5.0) < 0.021


def test_clients_differ():
    a = synth.fill(7, 0, 0, 1.0, "f32", 0, 1000)
    b = synth.fill(7, 1, 0, 1.0, "f32", 0, 1000)
    assert not np.array_equal(a, b)


@pytest.mark.parametrize("name,P,nk,K", [("tiny", 373386, 8, 4), ("unet3d", 18827472, 96, 10),
                                          ("lora", 16777216, 256, 8), ("vlm2b", 2205274112, 372, 8),
                                          ("llama7b", 6738415616, 291, 16)])
def test_workload_sizes(name, P, nk, K):
    w = W.make(name)
    assert (w.P, w.n_keys, w.K) == (P, nk, K)
    assert all(v == int(v) and 0 < v <= 2 ** 24 for v in w.weights)


def test_lora_reports_modules_in_pairs():
    w = W.make("lora")
    for r in w.reports:
        assert 64 * 2 <= len(r) <= 128 * 2
        s = set(r)
        assert all((2 * m in s) == (2 * m + 1 in s) for m in range(128))


def test_llama7b_weights_zipf_and_one_student_client():
    w = W.make("llama7b")
    assert sorted(w.weights, reverse=True)[0] == 5000.0
    assert min(w.weights) == round(5000 * 16 ** -1.2)
    assert w.dists.count(1) == 1
