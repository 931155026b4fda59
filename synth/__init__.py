"""Seeded synthetic inputs for FedAvg aggregation (tests and bench).

Input creation only.  The element values come from one counter-based
definition (see synth.c) implemented twice, for the host (C) and for the
device (CUDA); weights, masks and layouts come from `workloads`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import workloads  # noqa: F401
from .workloads import BF16, F32  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
HOST_SO = os.path.join(_BUILD, "libsynth.so")
DEV_SO = os.path.join(_BUILD, "libsynth_dev.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def build_commands():
    """(output, argv) pairs; the caller may run them in parallel."""
    os.makedirs(_BUILD, exist_ok=True)
    return [
        (HOST_SO, ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                   os.path.join(_HERE, "synth.c"), "-o", HOST_SO, "-lm"]),
        (DEV_SO, [NVCC, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                  "-gencode", "arch=compute_103a,code=sm_103a", "--fmad=false",
                  "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
                  os.path.join(_HERE, "synth_dev.cu"), "-o", DEV_SO]),
    ]


def build(device: bool = True) -> None:
    procs = []
    for out, cmd in build_commands():
        if not device and out == DEV_SO:
            continue
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    for cmd, p in procs:
        log = p.communicate()[0].decode(errors="replace")
        if p.returncode != 0:
            raise RuntimeError(f"synth build failed: {' '.join(cmd)}\n{log}")


_host = None
_dev = None


def host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_SO):
            build(device=False)
        lib = ctypes.CDLL(HOST_SO)
        u64, i32, f64, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_fill.argtypes = [u64, u64, i32, f64, i32, u64, u64, vp]
        lib.synth_fill.restype = None
        lib.synth_gather.argtypes = [u64, u64, i32, f64, i32, vp, u64, vp]
        lib.synth_gather.restype = None
        lib.synth_client_key.argtypes = [u64, u64]
        lib.synth_client_key.restype = u64
        lib.synth_value.argtypes = [u64, i32, f64, u64]
        lib.synth_value.restype = f64
        _host = lib
    return _host


def dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_SO):
            raise RuntimeError("synth device library not built: run __graft_entry__.build()")
        lib = ctypes.CDLL(DEV_SO)
        u64, i32, f64, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_dev_fill.argtypes = [u64, u64, i32, f64, i32, u64, u64, vp, vp]
        lib.synth_dev_fill.restype = i32
        _dev = lib
    return _dev


def _dtype_code(dtype: str) -> int:
    return 0 if dtype == F32 else 1


def np_dtype(dtype: str):
    return np.float32 if dtype == F32 else np.uint16


def fill(seed, client, dist, sigma, dtype, first, n, threads=None, out=None) -> np.ndarray:
    """Elements first..first+n-1 of client `client`'s stream (uint16 bits for bf16),
    into `out` if given (a contiguous array of n elements of the stored dtype)."""
    if out is None:
        out = np.empty(n, dtype=np_dtype(dtype))
    elif out.size != n or out.dtype != np.dtype(np_dtype(dtype)) or not out.flags.c_contiguous:
        raise ValueError("out must be a contiguous array of n elements of the stored dtype")
    lib = host_lib()
    code = _dtype_code(dtype)
    threads = threads or min(32, os.cpu_count() or 1)
    step = max(1 << 16, -(-n // threads))
    itemsize = out.itemsize
    base = out.ctypes.data

    def part(j0):
        m = min(step, n - j0)
        lib.synth_fill(seed, client, dist, sigma, code, first + j0, m, base + j0 * itemsize)

    if n <= step:
        if n:
            part(0)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(part, range(0, n, step)))
    return out


def gather(seed, client, dist, sigma, dtype, idx) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, dtype=np_dtype(dtype))
    host_lib().synth_gather(seed, client, dist, sigma, _dtype_code(dtype),
                            idx.ctypes.data, idx.size, out.ctypes.data)
    return out


def fill_device(seed, client, dist, sigma, dtype, first, n, ptr, stream=0) -> None:
    rc = dev_lib().synth_dev_fill(seed, client, dist, sigma, _dtype_code(dtype),
                                  first, n, ptr, stream)
    if rc != 0:
        raise RuntimeError("synth_dev_fill failed")


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Decode stored inputs to float64 (exact)."""
    if dtype == F32:
        return a.astype(np.float64)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------ workload helpers
def client_flat(w, k, first, n, threads=None, out=None) -> np.ndarray:
    """Client k's values for flat (unpadded, layout-order) elements first..first+n-1."""
    return fill(w.seed, k, w.dists[k], w.sigma, w.dtype_in, first, n, threads, out)


def client_key(w, k, p) -> np.ndarray:
    off = w.flat_offsets()[p]
    return client_flat(w, k, off, w.numels[p])


def client_gather(w, k, flat_idx) -> np.ndarray:
    return gather(w.seed, k, w.dists[k], w.sigma, w.dtype_in, flat_idx)


def client_fill_device(w, k, first, n, ptr, stream=0) -> None:
    fill_device(w.seed, k, w.dists[k], w.sigma, w.dtype_in, first, n, ptr, stream)
