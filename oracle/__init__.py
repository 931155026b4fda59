"""FedAvg oracle -- TEST INFRASTRUCTURE ONLY.

Plain fp64 CPU statement of server-side weighted aggregation (see
fedavg_oracle.c for the definition and the passages it follows).  Only the
tests, the smoke check and the bench's CPU-baseline leg may import this
package; the product path never does, and this package imports nothing from
the product.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(hand sums from the pages' definitions, exact rational arithmetic, library
routines, invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
SO = os.path.join(_BUILD, "libfedavg_oracle.so")

F32, BF16, F64 = "f32", "bf16", "f64"
_CODES = {F32: 0, BF16: 1, F64: 2}


def build_commands():
    os.makedirs(_BUILD, exist_ok=True)
    return [(SO, ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                  os.path.join(_HERE, "fedavg_oracle.c"), "-o", SO, "-lm"])]


def build() -> None:
    for out, cmd in build_commands():
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{r.stdout.decode()}")


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(SO):
            build()
        L = ctypes.CDLL(SO)
        u32, u64, i32, f64, vp = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.fo_bf16_rne.argtypes = [f64]
        L.fo_bf16_rne.restype = ctypes.c_uint16
        L.fo_f32_rn.argtypes = [f64]
        L.fo_f32_rn.restype = ctypes.c_float
        L.fo_fedavg_key.argtypes = [u32, vp, vp, vp, i32, u64, i32, vp, vp, vp]
        L.fo_fedavg_key.restype = i32
        L.fo_fedavg_key_f64.argtypes = [u32, vp, vp, vp, i32, u64, vp]
        L.fo_fedavg_key_f64.restype = i32
        L.fo_fedavg_apply_key.argtypes = [u32, vp, vp, vp, i32, u64, vp, f64, i32, vp, vp, vp]
        L.fo_fedavg_apply_key.restype = i32
        L.fo_bf16_rne_n.argtypes = [vp, u64, vp]
        L.fo_bf16_rne_n.restype = None
        L.fo_f32_rn_n.argtypes = [vp, u64, vp]
        L.fo_f32_rn_n.restype = None
        _lib = L
    return _lib


def _np_out(dtype):
    return np.float32 if dtype == F32 else np.uint16


def bf16_rne(y) -> np.ndarray:
    """fp64 -> bfloat16 bits, round to nearest, ties to even."""
    y = np.ascontiguousarray(y, dtype=np.float64).ravel()
    out = np.empty(y.size, np.uint16)
    lib().fo_bf16_rne_n(y.ctypes.data, y.size, out.ctypes.data)
    return out


def f32_rn(y) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float64).ravel()
    out = np.empty(y.size, np.float32)
    lib().fo_f32_rn_n(y.ctypes.data, y.size, out.ctypes.data)
    return out


def _prep(weights, reported, xs, dtype_in):
    K = len(weights)
    n = np.ascontiguousarray(weights, dtype=np.float64)
    rep = np.ascontiguousarray([1 if r else 0 for r in reported], dtype=np.uint8)
    want = {F32: np.float32, BF16: np.uint16, F64: np.float64}[dtype_in]
    numel = None
    arrs = []
    for k in range(K):
        if reported[k]:
            a = np.ascontiguousarray(xs[k])
            if a.dtype != want:
                raise TypeError(f"client {k}: expected {want}, got {a.dtype}")
            if numel is None:
                numel = a.size
            elif a.size != numel:
                raise ValueError("clients disagree on numel")
            arrs.append(a)
        else:
            arrs.append(None)
    if numel is None:
        numel = 0
    ptrs = (ctypes.c_void_p * K)(*[(a.ctypes.data if a is not None else None) for a in arrs])
    return K, n, rep, ptrs, arrs, numel


def fedavg_key(weights, reported, xs, dtype_in, dtype_out, out=None):
    """One key: returns (out_or_None, N_p, cnt_p).  `out` (if given) is left
    untouched when the key has no weight; the returned first item is None then.
    xs[k] holds client k's values (float32, or uint16 bf16 bits); entries of
    clients that did not report are ignored."""
    K, n, rep, ptrs, arrs, numel = _prep(weights, reported, xs, dtype_in)
    res = out if out is not None else np.empty(numel, _np_out(dtype_out))
    N = ctypes.c_double()
    cnt = ctypes.c_uint32()
    wrote = lib().fo_fedavg_key(K, n.ctypes.data, rep.ctypes.data, ptrs, _CODES[dtype_in], numel,
                                _CODES[dtype_out], res.ctypes.data, ctypes.byref(N), ctypes.byref(cnt))
    return (res if wrote else None), N.value, cnt.value


def fedavg_key_f64(weights, reported, xs, dtype_in):
    """One key before the output cast: the fp64 quotient, or None if N_p == 0."""
    K, n, rep, ptrs, arrs, numel = _prep(weights, reported, xs, dtype_in)
    y = np.empty(numel, np.float64)
    wrote = lib().fo_fedavg_key_f64(K, n.ctypes.data, rep.ctypes.data, ptrs, _CODES[dtype_in],
                                    numel, y.ctypes.data)
    return y if wrote else None


def fedavg_apply_key(weights, reported, xs, dtype_in, base, server_lr, dtype_out, out=None):
    """Delta round for one key: round(base + server_lr * weighted mean of xs).
    Returns (out_or_None, N_p, cnt_p); `base` holds dtype_out values."""
    K, n, rep, ptrs, arrs, numel = _prep(weights, reported, xs, dtype_in)
    b = np.ascontiguousarray(base)
    want = np.float32 if dtype_out == F32 else np.uint16
    if b.dtype != want or b.size != numel:
        raise TypeError("base must hold numel values of dtype_out")
    res = out if out is not None else np.empty(numel, _np_out(dtype_out))
    N = ctypes.c_double()
    cnt = ctypes.c_uint32()
    wrote = lib().fo_fedavg_apply_key(K, n.ctypes.data, rep.ctypes.data, ptrs, _CODES[dtype_in], numel,
                                      b.ctypes.data, float(server_lr), _CODES[dtype_out], res.ctypes.data,
                                      ctypes.byref(N), ctypes.byref(cnt))
    return (res if wrote else None), N.value, cnt.value


def hierarchical_f64(silos, weights, reported, xs, dtype_in):
    """Two-level weighted mean (silo means, then a mean of silo means weighted by each
    silo's total), all in fp64.  silos: list of client-index lists."""
    means, totals = [], []
    for members in silos:
        y = fedavg_key_f64([weights[k] for k in members], [reported[k] for k in members],
                           [xs[k] for k in members], dtype_in)
        n = sum(weights[k] for k in members if reported[k])
        means.append(y if y is not None else np.zeros(1))
        totals.append(n if y is not None else 0.0)
    rep = [t > 0 for t in totals]
    return fedavg_key_f64(totals, rep, means, F64)
