"""Server-side FedAvg aggregation on one GB300: Python binding of libfedavg.so.

Thin ctypes marshalling over the C ABI in include/fedavg.h; every function
has the C name and raises FedAvgError on a negative status.  All device work
happens in the library's CUDA kernels: there is no Python or CPU compute path,
and importing the binding without the built library fails loudly.

Pointers may be given as ints, as objects with .data_ptr() (torch tensors) or
as numpy arrays (host memory); streams as ints or objects with .cuda_stream.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfedavg.so")

FA_OK = 0
FA_ERR_ARG = -1
FA_ERR_RANGE = -2
FA_ERR_DTYPE = -3
FA_ERR_WEIGHT = -4
FA_ERR_INCOMPLETE = -5
FA_ERR_STATE = -6
FA_ERR_NOMEM = -7
FA_ERR_CUDA = -8
FA_ERR_TIMEOUT = -9
FA_ERR_INTERNAL = -10

FA_F32 = 0
FA_BF16 = 1
FA_KEY_FLAT = -1
FA_FLAT_OUT = 1
FA_STAGE_HOST = 2
FA_COMPENSATED = 4
FA_TEST_WAIT_EXPIRES = 0x80000000
FA_NOALLOC_MAX_ELEMS = 1 << 22

DTYPES = {"f32": FA_F32, "bf16": FA_BF16, FA_F32: FA_F32, FA_BF16: FA_BF16}


class fa_key(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("numel", ctypes.c_uint64)]


class fa_opts(ctypes.Structure):
    _fields_ = [("size", ctypes.c_uint32), ("ring_slots", ctypes.c_uint32),
                ("slot_bytes", ctypes.c_uint64), ("timeout_ms", ctypes.c_uint32),
                ("flags", ctypes.c_uint32)]


class fa_stats(ctypes.Structure):
    _fields_ = [("kernel_launches", ctypes.c_uint64), ("client_bytes", ctypes.c_uint64),
                ("h2d_bytes", ctypes.c_uint64), ("d2h_bytes", ctypes.c_uint64),
                ("chunks", ctypes.c_uint64)]


class fa_partition_opts(ctypes.Structure):
    _fields_ = [("w_time", ctypes.c_double), ("w_energy", ctypes.c_double),
                ("ema_alpha", ctypes.c_double), ("deadband", ctypes.c_double)]


class FedAvgError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"{status} ({fa_strerror(status)}): {detail}")


_lib = None


def lib():
    """The loaded libfedavg.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        i32, u32, u64, i64, f64, vp = (ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64,
                                       ctypes.c_int64, ctypes.c_double, ctypes.c_void_p)
        L.fa_open.argtypes = [ctypes.POINTER(fa_key), u32, i32, i32, u32, ctypes.POINTER(fa_opts),
                              ctypes.POINTER(vp)]
        L.fa_accumulate.argtypes = [vp, u32, f64, i64, u64, vp, u64, vp]
        L.fa_accumulate_batch.argtypes = [vp, u32, ctypes.POINTER(u32), ctypes.POINTER(f64), i64,
                                          u64, ctypes.POINTER(vp), u64, vp]
        L.fa_accumulate_keys.argtypes = [vp, u32, f64, u32, ctypes.POINTER(i64), ctypes.POINTER(u64),
                                         ctypes.POINTER(vp), ctypes.POINTER(u64), vp]
        L.fa_accumulate_final.argtypes = [vp, u32, f64, i64, u64, vp, u64, ctypes.POINTER(vp), vp]
        L.fa_finalize.argtypes = [vp, ctypes.POINTER(vp), vp]
        L.fa_reduce_resident.argtypes = [vp, u32, ctypes.POINTER(u32), ctypes.POINTER(f64),
                                         ctypes.POINTER(vp), ctypes.POINTER(vp), vp]
        L.fa_finalize_apply.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), f64, vp]
        L.fa_reduce_subsets.argtypes = [vp, u32, ctypes.POINTER(u32), ctypes.POINTER(f64),
                                        ctypes.POINTER(vp), ctypes.POINTER(u32), ctypes.POINTER(i64),
                                        ctypes.POINTER(vp), vp]
        L.fa_reset.argtypes = [vp]
        L.fa_close.argtypes = [vp]
        L.fa_key_total.argtypes = [vp, u32, ctypes.POINTER(f64), ctypes.POINTER(u32)]
        L.fa_sync.argtypes = [vp]
        L.fa_get_stats.argtypes = [vp, ctypes.POINTER(fa_stats)]
        L.fa_aggregate_noalloc.argtypes = [u32, ctypes.POINTER(f64), ctypes.POINTER(vp), u64, i32, i32,
                                           vp, vp]
        L.fa_aggregate_noalloc.restype = i32
        L.fa_aggregate_noalloc_status.argtypes = [vp, u32]
        L.fa_aggregate_noalloc_status.restype = i32
        L.fa_partition_plan.argtypes = [u32, vp, vp, vp, vp, vp, ctypes.POINTER(fa_partition_opts), vp]
        L.fa_partition_plan.restype = i32
        L.fa_strerror.argtypes = [i32]
        L.fa_strerror.restype = ctypes.c_char_p
        L.fa_last_error.argtypes = [vp]
        L.fa_last_error.restype = ctypes.c_char_p
        for name in ("fa_open", "fa_accumulate", "fa_accumulate_batch", "fa_accumulate_keys",
                     "fa_accumulate_final", "fa_finalize",
                     "fa_finalize_apply", "fa_reduce_resident", "fa_reduce_subsets", "fa_reset",
                     "fa_close", "fa_key_total", "fa_sync", "fa_get_stats"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):
        return int(x.ctypes.data)
    raise TypeError(f"cannot take a pointer of {type(x)!r}")


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(status: int, ctx=None):
    if status != FA_OK:
        detail = fa_last_error(ctx) if ctx is not None else ""
        raise FedAvgError(status, detail)


def fa_strerror(status: int) -> str:
    return lib().fa_strerror(status).decode()


def fa_last_error(ctx) -> str:
    r = lib().fa_last_error(ctx)
    return r.decode() if r else ""


def fa_open(layout, dtype_in, dtype_out, max_clients, ring_slots=0, slot_bytes=0,
            timeout_ms=0, flags=0):
    """layout: list of (name, numel).  Returns an opaque context handle."""
    n = len(layout)
    keys = (fa_key * max(n, 1))()
    names = []
    for i, (name, numel) in enumerate(layout):
        b = name.encode() if isinstance(name, str) else name
        names.append(b)
        keys[i].name = b
        keys[i].numel = int(numel)
    opts = fa_opts(ctypes.sizeof(fa_opts), ring_slots, slot_bytes, timeout_ms, flags)
    ctx = ctypes.c_void_p()
    _check(lib().fa_open(keys, n, DTYPES[dtype_in], DTYPES[dtype_out], max_clients,
                         ctypes.byref(opts), ctypes.byref(ctx)))
    return ctx


def fa_accumulate(ctx, client_id, weight_nk, key, offset_elems, chunk, len_elems, stream=None):
    _check(lib().fa_accumulate(ctx, client_id, float(weight_nk), key, offset_elems, _ptr(chunk),
                               len_elems, _stream(stream)), ctx)


def out_array(outs):
    """A C array of output pointers (per-key outputs, None allowed, or one flat output)."""
    return (ctypes.c_void_p * max(len(outs), 1))(*[_ptr(o) for o in outs])


def fa_accumulate_final(ctx, client_id, weight_nk, key, offset_elems, chunk, len_elems, outs,
                        stream=None):
    """outs: as for fa_finalize, or an array made by out_array (reused across calls)."""
    ps = outs if isinstance(outs, ctypes.Array) else out_array(outs)
    _check(lib().fa_accumulate_final(ctx, client_id, float(weight_nk), key, offset_elems, _ptr(chunk),
                                     len_elems, ps, _stream(stream)), ctx)


def _same_length(**seqs):
    n = {k: len(v) for k, v in seqs.items()}
    if len(set(n.values())) > 1:
        raise ValueError("lengths differ: " + ", ".join(f"{k}={v}" for k, v in n.items()))


def fa_accumulate_batch(ctx, client_ids, weights, key, offset_elems, chunks, len_elems,
                        stream=None):
    _same_length(client_ids=client_ids, weights=weights, chunks=chunks)
    J = len(client_ids)
    ids = (ctypes.c_uint32 * J)(*client_ids)
    ws = (ctypes.c_double * J)(*[float(w) for w in weights])
    ps = (ctypes.c_void_p * J)(*[_ptr(c) for c in chunks])
    _check(lib().fa_accumulate_batch(ctx, J, ids, ws, key, offset_elems, ps, len_elems,
                                     _stream(stream)), ctx)


def fa_accumulate_keys(ctx, client_id, weight_nk, keys, offsets, chunks, lens, stream=None):
    """One client's chunks in one call: chunk i is `lens[i]` elements at `offsets[i]` of
    key `keys[i]` (FA_KEY_FLAT: of the flat layout), read from `chunks[i]` (pointers as
    ints or a uint64 array, or tensors / arrays).  Sequences or NumPy arrays."""
    import numpy as np
    ks = np.ascontiguousarray(keys, dtype=np.int64)
    os_ = np.ascontiguousarray(offsets, dtype=np.uint64)
    ls = np.ascontiguousarray(lens, dtype=np.uint64)
    if isinstance(chunks, np.ndarray):
        ps = np.ascontiguousarray(chunks, dtype=np.uint64)
    else:
        ps = np.fromiter((_ptr(c) for c in chunks), dtype=np.uint64, count=len(chunks))
    n = ks.size
    if not (os_.size == ps.size == ls.size == n):
        raise ValueError("keys, offsets, chunks and lens must have the same length")
    _check(lib().fa_accumulate_keys(
        ctx, client_id, float(weight_nk), n, ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        os_.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
        ps.ctypes.data_as(ctypes.POINTER(ctypes.c_void_p)),
        ls.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), _stream(stream)), ctx)


def fa_finalize(ctx, outs, stream=None):
    """outs: list of per-key outputs (None allowed for keys that will not be written),
    or a one-element list with the flat output when opened with FA_FLAT_OUT."""
    ps = (ctypes.c_void_p * max(len(outs), 1))(*[_ptr(o) for o in outs])
    _check(lib().fa_finalize(ctx, ps, _stream(stream)), ctx)


def fa_finalize_apply(ctx, bases, outs, server_lr=1.0, stream=None):
    """Delta rounds: outs = round(bases + server_lr * weighted mean); outs may be bases."""
    bs = (ctypes.c_void_p * max(len(bases), 1))(*[_ptr(b) for b in bases])
    ps = (ctypes.c_void_p * max(len(outs), 1))(*[_ptr(o) for o in outs])
    _check(lib().fa_finalize_apply(ctx, bs, ps, float(server_lr), _stream(stream)), ctx)


def fa_reduce_resident(ctx, client_ids, weights, flat_updates, outs, stream=None):
    """Whole round from resident full updates (one flat buffer per client) straight to outs."""
    _same_length(client_ids=client_ids, weights=weights, flat_updates=flat_updates)
    J = len(client_ids)
    ids = (ctypes.c_uint32 * J)(*client_ids)
    ws = (ctypes.c_double * J)(*[float(w) for w in weights])
    ps = (ctypes.c_void_p * J)(*[_ptr(x) for x in flat_updates])
    os_ = (ctypes.c_void_p * max(len(outs), 1))(*[_ptr(o) for o in outs])
    _check(lib().fa_reduce_resident(ctx, J, ids, ws, ps, os_, _stream(stream)), ctx)


def subset_table(client_keys):
    """Marshal per-client key lists once: (n_keys uint32 array, concatenated int64 keys)."""
    import numpy as np
    nk = np.ascontiguousarray([len(k) for k in client_keys], dtype=np.uint32)
    ks = np.ascontiguousarray(np.concatenate([np.asarray(k, np.int64) for k in client_keys])
                              if len(client_keys) else np.zeros(0, np.int64), dtype=np.int64)
    return nk, ks


def fa_reduce_subsets(ctx, client_ids, weights, client_bufs, client_keys, outs, stream=None):
    """A round of key subsets resident in device memory, straight to outs: client j's
    buffer client_bufs[j] holds its keys client_keys[j] (a list of key ids) packed back to
    back in that order.  client_keys may also be a subset_table(...) result."""
    import numpy as np
    if isinstance(client_keys, tuple) and len(client_keys) == 2 and isinstance(client_keys[0], np.ndarray):
        nk, ks = client_keys
        _same_length(client_ids=client_ids, weights=weights, client_bufs=client_bufs, n_keys=nk)
    else:
        _same_length(client_ids=client_ids, weights=weights, client_bufs=client_bufs,
                     client_keys=client_keys)
        nk, ks = subset_table(client_keys)
    J = len(client_ids)
    ids = (ctypes.c_uint32 * J)(*client_ids)
    ws = (ctypes.c_double * J)(*[float(w) for w in weights])
    ps = (ctypes.c_void_p * J)(*[_ptr(b) for b in client_bufs])
    os_ = (ctypes.c_void_p * max(len(outs), 1))(*[_ptr(o) for o in outs])
    _check(lib().fa_reduce_subsets(ctx, J, ids, ws, ps, nk.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)),
                                   ks.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), os_,
                                   _stream(stream)), ctx)


def fa_reset(ctx):
    _check(lib().fa_reset(ctx), ctx)


def fa_close(ctx):
    _check(lib().fa_close(ctx))


def fa_key_total(ctx, key):
    s = ctypes.c_double()
    n = ctypes.c_uint32()
    _check(lib().fa_key_total(ctx, key, ctypes.byref(s), ctypes.byref(n)), ctx)
    return s.value, n.value


def fa_sync(ctx):
    _check(lib().fa_sync(ctx), ctx)


def fa_get_stats(ctx) -> dict:
    st = fa_stats()
    _check(lib().fa_get_stats(ctx, ctypes.byref(st)), ctx)
    return {f: getattr(st, f) for f, _ in fa_stats._fields_}


def fa_aggregate_noalloc(weights, chunks, numel, dtype_in, dtype_out, out, stream=None):
    """One tensor, all clients resident, no allocation: the running sum lives in a
    fixed 16 MiB array of the library (see include/fedavg.h).  For callers that must
    not have a library allocate device memory."""
    _same_length(weights=weights, chunks=chunks)
    J = len(chunks)
    ws = (ctypes.c_double * max(J, 1))(*[float(w) for w in weights])
    ps = (ctypes.c_void_p * max(J, 1))(*[_ptr(c) for c in chunks])
    _check(lib().fa_aggregate_noalloc(J, ws, ps, numel, DTYPES[dtype_in], DTYPES[dtype_out],
                                      _ptr(out), _stream(stream)))


def fa_aggregate_noalloc_status(stream=None, timeout_ms=0):
    """Raises FedAvgError (FA_ERR_INTERNAL) if a device-side wait gave up in an
    fa_aggregate_noalloc call on the current device since the last check."""
    _check(lib().fa_aggregate_noalloc_status(_stream(stream), timeout_ms))


def fa_partition_plan(time_s, energy_j, samples, ema_tau=None, ema_eps=None, w_time=1.0,
                      w_energy=0.0, ema_alpha=0.5, deadband=0.05):
    """Next round's sample counts; returns (new_samples, ema_tau, ema_eps) as lists."""
    import numpy as np
    m = len(samples)
    t = np.ascontiguousarray(time_s, dtype=np.float64)
    e = np.ascontiguousarray(energy_j, dtype=np.float64)
    n = np.ascontiguousarray(samples, dtype=np.uint64)
    tau = np.full(m, np.nan) if ema_tau is None else np.array(ema_tau, dtype=np.float64)
    eps = np.full(m, np.nan) if ema_eps is None else np.array(ema_eps, dtype=np.float64)
    out = np.zeros(m, dtype=np.uint64)
    o = fa_partition_opts(w_time, w_energy, ema_alpha, deadband)
    _check(lib().fa_partition_plan(m, t.ctypes.data, e.ctypes.data, n.ctypes.data, tau.ctypes.data,
                                   eps.ctypes.data, ctypes.byref(o), out.ctypes.data))
    return [int(v) for v in out], tau.tolist(), eps.tolist()
