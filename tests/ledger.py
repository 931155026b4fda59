"""ctypes wrapper of the host-only ledger shim (tests/native/ledger_shim.cpp)."""
import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "server_side_fedavg_gb300", "csrc")
SO = os.path.join(HERE, "_build", "libledger_shim.so")

_lib = None


def lib():
    global _lib
    if _lib is None:
        os.makedirs(os.path.dirname(SO), exist_ok=True)
        srcs = [os.path.join(HERE, "native", "ledger_shim.cpp"), os.path.join(CSRC, "ledger.cpp")]
        if not os.path.exists(SO) or any(os.path.getmtime(s) > os.path.getmtime(SO) for s in srcs):
            subprocess.run(["g++", "-O1", "-g", "-std=c++17", "-fPIC", "-shared", "-I", CSRC] + srcs
                           + ["-o", SO], check=True)
        L = ctypes.CDLL(SO)
        u32, u64, i32, i64, f64, vp = (ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32,
                                       ctypes.c_int64, ctypes.c_double, ctypes.c_void_p)
        L.lg_new.argtypes = [vp, u32, u32, ctypes.POINTER(i32)]
        L.lg_new.restype = vp
        L.lg_free.argtypes = [vp]
        L.lg_error.argtypes = [vp]
        L.lg_error.restype = ctypes.c_char_p
        L.lg_accumulate.argtypes = [vp, vp, vp, u32, i64, u64, u64, vp, u32, ctypes.POINTER(u32)]
        L.lg_accumulate.restype = i32
        L.lg_accumulate_keys.argtypes = [vp, u32, f64, u32, vp, vp, vp, vp, u32, ctypes.POINTER(u32)]
        L.lg_accumulate_keys.restype = i32
        L.lg_whole_keys.argtypes = [vp, u32, f64, u32, vp]
        L.lg_whole_keys.restype = i32
        L.lg_finalize.argtypes = [vp, vp, vp, u32, ctypes.POINTER(u32)]
        L.lg_finalize.restype = i32
        L.lg_reset.argtypes = [vp]
        L.lg_key_total.argtypes = [vp, u32, ctypes.POINTER(f64), ctypes.POINTER(u32)]
        L.lg_key_total.restype = i32
        L.lg_accumulate_final.argtypes = [vp, u32, f64, i64, u64, u64, vp, vp, u32, ctypes.POINTER(u32)]
        L.lg_accumulate_final.restype = i32
        L.lg_finalize_ranges.argtypes = [vp, vp, vp, u32, ctypes.POINTER(u32)]
        L.lg_finalize_ranges.restype = i32
        L.lg_has_final.argtypes = [vp]
        L.lg_has_final.restype = i32
        L.lg_acc_off.argtypes = [vp, u32]
        L.lg_acc_off.restype = u64
        L.lg_padded.argtypes = [vp]
        L.lg_padded.restype = u64
        _lib = L
    return _lib


class Ledger:
    def __init__(self, numels, max_clients):
        arr = (ctypes.c_uint64 * len(numels))(*numels)
        st = ctypes.c_int32()
        self.h = lib().lg_new(arr, len(numels), max_clients, ctypes.byref(st))
        self.status = st.value
        self.n_keys = len(numels)

    def __del__(self):
        if getattr(self, "h", None):
            lib().lg_free(self.h)

    def error(self):
        return lib().lg_error(self.h).decode()

    def accumulate(self, clients, weights, key, offset, length):
        J = len(clients)
        c = (ctypes.c_uint32 * J)(*clients)
        w = (ctypes.c_double * J)(*weights)
        rows = (ctypes.c_uint64 * (5 * 4096))()
        n = ctypes.c_uint32()
        st = lib().lg_accumulate(self.h, c, w, J, key, offset, length, rows, 4096, ctypes.byref(n))
        pieces = [tuple(rows[5 * i:5 * i + 5]) for i in range(min(n.value, 4096))]
        return st, pieces

    def accumulate_keys(self, client, weight, chunks):
        """chunks: [(key, offset, length)] of one client.  Returns (status, pieces) with
        pieces as (chunk, key, chunk_off, acc_idx, len, first)."""
        n = len(chunks)
        keys = (ctypes.c_int64 * max(n, 1))(*[c[0] for c in chunks])
        offs = (ctypes.c_uint64 * max(n, 1))(*[c[1] for c in chunks])
        lens = (ctypes.c_uint64 * max(n, 1))(*[c[2] for c in chunks])
        rows = (ctypes.c_uint64 * (6 * 4096))()
        m = ctypes.c_uint32()
        st = lib().lg_accumulate_keys(self.h, client, weight, n, keys, offs, lens, rows, 4096,
                                      ctypes.byref(m))
        return st, [tuple(rows[6 * i:6 * i + 6]) for i in range(min(m.value, 4096))]

    def whole_keys(self, client, weight, keys):
        n = len(keys)
        ks = (ctypes.c_int64 * max(n, 1))(*keys)
        return lib().lg_whole_keys(self.h, client, weight, n, ks)

    def finalize(self):
        rows = (ctypes.c_uint64 * (5 * 4096))()
        tot = (ctypes.c_double * 4096)()
        n = ctypes.c_uint32()
        st = lib().lg_finalize(self.h, rows, tot, 4096, ctypes.byref(n))
        items = [tuple(rows[5 * i:5 * i + 5]) + (tot[i],) for i in range(min(n.value, 4096))]
        return st, items

    def accumulate_final(self, client, weight, key, offset, length):
        """Returns (status, pieces as in accumulate, each piece's N_p)."""
        rows = (ctypes.c_uint64 * (5 * 4096))()
        tot = (ctypes.c_double * 4096)()
        n = ctypes.c_uint32()
        st = lib().lg_accumulate_final(self.h, client, weight, key, offset, length, rows, tot, 4096,
                                       ctypes.byref(n))
        m = min(n.value, 4096)
        return st, [tuple(rows[5 * i:5 * i + 5]) for i in range(m)], [tot[i] for i in range(m)]

    def finalize_ranges(self):
        """The ranges fa_finalize would write, without closing the round: (status,
        [(key, koff, acc_idx, flat_off, numel, reporters, total)])."""
        rows = (ctypes.c_uint64 * (6 * 4096))()
        tot = (ctypes.c_double * 4096)()
        n = ctypes.c_uint32()
        st = lib().lg_finalize_ranges(self.h, rows, tot, 4096, ctypes.byref(n))
        return st, [tuple(rows[6 * i:6 * i + 6]) + (tot[i],) for i in range(min(n.value, 4096))]

    def has_final(self):
        """Whether a final contribution has written a range this round."""
        return bool(lib().lg_has_final(self.h))

    def reset(self):
        lib().lg_reset(self.h)

    def key_total(self, key):
        t = ctypes.c_double()
        r = ctypes.c_uint32()
        st = lib().lg_key_total(self.h, key, ctypes.byref(t), ctypes.byref(r))
        return st, t.value, r.value

    def acc_off(self, key):
        return lib().lg_acc_off(self.h, key)

    def padded(self):
        return lib().lg_padded(self.h)
