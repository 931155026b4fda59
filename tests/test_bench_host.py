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


def test_byte_counts_of_the_streamed_round():
    """The 7B round's algorithmic bytes: unfused 6 + 15 * 10 + 6 bytes per element
    (1,091.6 GB); fused 6 + 14 * 10 + 8 (1,037.7 GB), its plain launches (clients 0..14,
    765 launches of 256 MiB flat chunks) 1,286,024,418 bytes each on average and the last
    client's 51 final-form launches 8 bytes per element."""
    w = W.make("llama7b")
    P = w.P
    first, later, fin = bench.algorithmic_bytes(w)
    assert (first, later, fin) == (6 * P, 15 * 10 * P, 6 * P)
    assert first + later + fin == 1_091_623_329_792
    b0, b1, b2 = bench.fused_bytes(w)
    assert (b0, b1, b2) == (6 * P, 14 * 10 * P, 8 * P)
    assert b0 + b1 + b2 == 1_037_716_004_864
    nchunk = -(-P // w.chunk_elems)
    assert nchunk == 51
    assert (b0 + b1) // ((w.K - 1) * nchunk) == 1_286_024_418
