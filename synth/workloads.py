"""Synthetic FedAvg workloads: layouts, client weights, participation masks.

Input creation only: nothing here averages, divides or rounds an aggregate.
Every quantity is a pure function of the workload's seed, so the CUDA path
and the oracle see the same inputs.

Workloads (shapes and distributions follow the federated-learning pages:
the FLARE multimodal blog's full-model and adapter-only (FedUMM) updates,
the Clara Train FL article's BRATS brain-tumour segmentation model, and the
adaptive-partitioning summary's per-participant sample counts n_i):

  tiny      K=4,  8 fp32 tensors of a small CNN, N(0,0.05), n_k ~ U{100..1000}
  unet3d    K=10, 96 fp32 tensors of a 3-D U-Net (3x3x3 convs), deltas N(0,1e-3),
            n_k = round(exp(U(ln 50, ln 5000)))
  lora      K=8,  bf16 rank-16 LoRA A/B on q,k,v,o of 32 layers, each client
            reports a seeded random 64..128 of the 128 modules, N(0,0.01)
  vlm2b     K=8,  2.2B-parameter VLM-shaped bf16 state dict, N(0,0.02),
            streamed in 64 MiB flat chunks
  llama7b   K=16, 7B-parameter decoder bf16 state dict, N(0,0.02) except one
            seeded client at 0.02*Student-t(3); n_k Zipf(1.2)-skewed;
            streamed in 256 MiB flat chunks
  decoder1l K=4, one layer of the 7B decoder (profiling size)
  mlp16     K=16, gate and up projections of one 7B layer (profiling size)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

from . import _rng

F32 = "f32"
BF16 = "bf16"
DIST_NORMAL = 0
DIST_STUDENT3 = 1

BASE_SEED = 20261202


@dataclass
class Workload:
    name: str
    index: int
    keys: list            # [(name, shape tuple)]
    K: int
    dtype_in: str
    dtype_out: str
    sigma: float
    weights: list         # n_k, float (integer-valued)
    reports: list         # reports[k] = sorted list of key indices client k sends
    dists: list           # per client DIST_*
    chunk_elems: int      # flat streaming chunk (0 = one chunk per tensor)
    seed: int = 0
    numels: list = field(default_factory=list)

    @property
    def P(self) -> int:
        return sum(self.numels)

    @property
    def n_keys(self) -> int:
        return len(self.keys)

    def flat_offsets(self):
        """Start of each key in the unpadded concatenation (layout order)."""
        out, o = [], 0
        for n in self.numels:
            out.append(o)
            o += n
        return out

    def client_bytes(self) -> int:
        s = 2 if self.dtype_in == BF16 else 4
        return sum(self.numels[p] for k in range(self.K) for p in self.reports[k]) * s


def _numel(shape):
    n = 1
    for d in shape:
        n *= d
    return n


def _finish(w: Workload) -> Workload:
    w.numels = [_numel(s) for _, s in w.keys]
    return w


# ---------------------------------------------------------------- layouts
def tiny_layout():
    return [("conv1.weight", (64, 3, 3, 3)), ("conv1.bias", (64,)),
            ("conv2.weight", (128, 64, 3, 3)), ("conv2.bias", (128,)),
            ("conv3.weight", (256, 128, 3, 3)), ("conv3.bias", (256,)),
            ("fc.weight", (10, 256)), ("fc.bias", (10,))]


UNET_BLOCKS = [(4, 32), (32, 32), (32, 64), (64, 64), (64, 128), (128, 128),
               (128, 256), (256, 256), (256, 256), (256, 256), (256, 256),
               (256, 256), (512, 256), (256, 256), (256, 128), (256, 128),
               (128, 128), (128, 64), (128, 64), (64, 64), (64, 32), (64, 32),
               (32, 32), (32, 16)]


def unet3d_layout():
    keys = []
    for b, (cin, cout) in enumerate(UNET_BLOCKS):
        keys += [(f"block{b}.conv.weight", (cout, cin, 3, 3, 3)),
                 (f"block{b}.conv.bias", (cout,)),
                 (f"block{b}.norm.weight", (cout,)),
                 (f"block{b}.norm.bias", (cout,))]
    return keys


def lora_layout(layers=32, hidden=4096, rank=16):
    keys = []
    for l in range(layers):
        for m in ("q_proj", "k_proj", "v_proj", "o_proj"):
            keys.append((f"layers.{l}.{m}.lora_A", (rank, hidden)))
            keys.append((f"layers.{l}.{m}.lora_B", (hidden, rank)))
    return keys


def vlm2b_layout():
    h, f, v = 4096, 11008, 32000
    keys = [("lm.embed_tokens", (v, h))]
    for l in range(8):
        p = f"lm.layers.{l}."
        keys += [(p + "q_proj", (h, h)), (p + "k_proj", (h, h)),
                 (p + "v_proj", (h, h)), (p + "o_proj", (h, h)),
                 (p + "gate_proj", (f, h)), (p + "up_proj", (f, h)),
                 (p + "down_proj", (h, f)),
                 (p + "input_norm", (h,)), (p + "post_norm", (h,))]
    keys += [("lm.norm", (h,)), ("lm.lm_head", (v, h))]
    d, m = 1024, 4096
    for l in range(24):
        p = f"vit.layers.{l}."
        keys += [(p + "q_proj", (d, d)), (p + "k_proj", (d, d)),
                 (p + "v_proj", (d, d)), (p + "o_proj", (d, d)),
                 (p + "fc1.weight", (m, d)), (p + "fc1.bias", (m,)),
                 (p + "fc2.weight", (d, m)), (p + "fc2.bias", (d,)),
                 (p + "ln1.weight", (d,)), (p + "ln1.bias", (d,)),
                 (p + "ln2.weight", (d,)), (p + "ln2.bias", (d,))]
    keys += [("vit.patch_embed.weight", (d, 3, 14, 14)), ("vit.patch_embed.bias", (d,)),
             ("vit.pos_embed", (257, d)),
             ("vit.post_ln.weight", (d,)), ("vit.post_ln.bias", (d,)),
             ("projector.0.weight", (h, d)), ("projector.0.bias", (h,)),
             ("projector.2.weight", (h, h)), ("projector.2.bias", (h,))]
    return keys


def llama7b_layout(layers=32):
    h, f, v = 4096, 11008, 32000
    keys = [("embed_tokens", (v, h))]
    for l in range(layers):
        p = f"layers.{l}."
        keys += [(p + "q_proj", (h, h)), (p + "k_proj", (h, h)),
                 (p + "v_proj", (h, h)), (p + "o_proj", (h, h)),
                 (p + "gate_proj", (f, h)), (p + "up_proj", (f, h)),
                 (p + "down_proj", (h, f)),
                 (p + "input_norm", (h,)), (p + "post_norm", (h,))]
    keys += [("norm", (h,)), ("lm_head", (v, h))]
    return keys


# ---------------------------------------------------------------- weights / masks
def uniform_int_weights(seed, K, lo=100, hi=1000):
    return [float(lo + _rng.below(seed, 1000 + k, hi - lo + 1)) for k in range(K)]


def loguniform_weights(seed, K, lo=50.0, hi=5000.0):
    out = []
    for k in range(K):
        u = _rng.unit(seed, 2000 + k)
        out.append(float(round(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))))
    return out


def zipf_weights(seed, K, top=5000.0, s=1.2):
    ranks = _rng.permutation(seed, 3000, K)          # a permutation of 0..K-1
    return [float(round(top * (r + 1) ** (-s))) for r in ranks]


def lora_reports(seed, K, n_modules=128, lo=64, hi=128):
    reports = []
    for k in range(K):
        m = lo + _rng.below(seed, 4000 + k, hi - lo + 1)
        perm = _rng.permutation(seed, 5000 + k, n_modules)
        mods = sorted(perm[:m])
        keys = []
        for mod in mods:          # A and B of a module travel together
            keys += [2 * mod, 2 * mod + 1]
        reports.append(keys)
    return reports


# ---------------------------------------------------------------- the five workloads
def make(name: str) -> Workload:
    if name == "tiny":
        i = 0
        seed = BASE_SEED + i
        keys = tiny_layout()
        K = 4
        w = Workload(name, i, keys, K, F32, F32, 0.05, uniform_int_weights(seed, K),
                     [list(range(len(keys)))] * K, [DIST_NORMAL] * K, 0, seed)
    elif name == "unet3d":
        i = 1
        seed = BASE_SEED + i
        keys = unet3d_layout()
        K = 10
        w = Workload(name, i, keys, K, F32, F32, 1e-3, loguniform_weights(seed, K),
                     [list(range(len(keys)))] * K, [DIST_NORMAL] * K, 0, seed)
    elif name == "lora":
        i = 2
        seed = BASE_SEED + i
        keys = lora_layout()
        K = 8
        w = Workload(name, i, keys, K, BF16, BF16, 0.01, uniform_int_weights(seed, K),
                     lora_reports(seed, K), [DIST_NORMAL] * K, 0, seed)
    elif name == "vlm2b":
        i = 3
        seed = BASE_SEED + i
        keys = vlm2b_layout()
        K = 8
        w = Workload(name, i, keys, K, BF16, BF16, 0.02, uniform_int_weights(seed, K),
                     [list(range(len(keys)))] * K, [DIST_NORMAL] * K,
                     (64 << 20) // 2, seed)
    elif name == "llama7b":
        i = 4
        seed = BASE_SEED + i
        keys = llama7b_layout()
        K = 16
        dists = [DIST_NORMAL] * K
        dists[_rng.below(seed, 6000, K)] = DIST_STUDENT3
        w = Workload(name, i, keys, K, BF16, BF16, 0.02, zipf_weights(seed, K),
                     [list(range(len(keys)))] * K, dists, (256 << 20) // 2, seed)
    elif name == "decoder1l":
        # one decoder layer of the 7B shape, K=4: the same kernels and chunking as
        # llama7b at about 3 GB of device memory, still far larger than L2
        i = 5
        seed = BASE_SEED + i
        keys = llama7b_layout(layers=1)[1:10]
        K = 4
        w = Workload(name, i, keys, K, BF16, BF16, 0.02, uniform_int_weights(seed, K),
                     [list(range(len(keys)))] * K, [DIST_NORMAL] * K, (256 << 20) // 2, seed)
    elif name == "mlp16":
        # the gate and up projections of one 7B decoder layer, K=16 clients all resident:
        # the resident-reduce kernels of llama7b at about 3.4 GB of device memory
        i = 6
        seed = BASE_SEED + i
        keys = llama7b_layout(layers=1)[5:7]
        K = 16
        w = Workload(name, i, keys, K, BF16, BF16, 0.02, uniform_int_weights(seed, K),
                     [list(range(len(keys)))] * K, [DIST_NORMAL] * K, (256 << 20) // 2, seed)
    else:
        raise ValueError(f"unknown workload {name!r}")
    return _finish(w)


NAMES = ("tiny", "unet3d", "lora", "vlm2b", "llama7b")
EXTRA = ("decoder1l", "mlp16")
