"""Host-side helpers of bench.py: which kernel fa_reduce_resident runs for each workload
(the library's rule: more than 48 keys from at most 16 clients, with per-key tables that fit
a launch's parameters, take the one-launch subset-reduce kernel)."""
import bench
from synth import workloads as W


def test_resident_kernel_per_workload():
    assert bench.resident_kernel(W.make("unet3d")).startswith("reduce_gather_inline_kernel")
    for name in ("tiny", "llama7b", "vlm2b", "mlp16", "decoder1l"):
        assert bench.resident_kernel(W.make(name)).startswith("reduce_bulk_kernel"), name


def test_subsets_kernel_for_the_lora_round():
    assert bench.subsets_kernel(W.make("lora")).startswith("reduce_gather_inline_kernel")
