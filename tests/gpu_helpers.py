"""Device-side helpers shared by the GPU tests (torch for memory and streams only)."""
import numpy as np
import torch

import server_side_fedavg_gb300 as fa


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def to_dev(x: np.ndarray) -> torch.Tensor:
    if x.dtype == np.uint16:
        x = x.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev())


def to_pinned(x: np.ndarray) -> torch.Tensor:
    if x.dtype == np.uint16:
        x = x.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(x)).pin_memory()


def to_np(t: torch.Tensor, dtype: str) -> np.ndarray:
    a = t.detach().cpu().numpy()
    return a.view(np.uint16) if dtype == "bf16" else a


def torch_dtype(dtype: str):
    return torch.float32 if dtype == "f32" else torch.int16


def sentinel(n: int, dtype: str, device=None) -> torch.Tensor:
    """A recognisable pattern for 'not written' checks (fp32 -7.0 / bf16 0x7FBF)."""
    if dtype == "f32":
        return torch.full((n,), -7.0, dtype=torch.float32, device=device or dev())
    return torch.full((n,), 0x7FBF, dtype=torch.int16, device=device or dev())


def sentinel_np(n: int, dtype: str) -> np.ndarray:
    return to_np(sentinel(n, dtype, device="cpu"), dtype)


def ragged_splits(n: int, pieces: int, rng) -> list:
    """Split [0, n) into `pieces` contiguous ragged ranges (some may be tiny)."""
    if pieces <= 1 or n < pieces:
        return [(0, n)]
    cuts = sorted(set(int(c) for c in rng.integers(1, n, pieces - 1)))
    b = [0] + cuts + [n]
    return [(b[i], b[i + 1]) for i in range(len(b) - 1)]
