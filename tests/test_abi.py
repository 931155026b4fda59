"""The C ABI library loads and exports every entry point include/fedavg.h
declares, its constants agree with the binding, and argument errors that need
no device come back as status codes (CPU; no compute calls)."""
import ctypes
import os
import re

import pytest

import server_side_fedavg_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fedavg.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def _defines():
    out = {}
    for m in re.finditer(r"#define\s+(FA_\w+)\s+\(?(-?\w+)\)?", open(HEADER).read()):
        try:
            out[m.group(1)] = int(m.group(2).rstrip("uU"), 0)
        except ValueError:
            pass
    return out


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return fa.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in fedavg.h but not exported"


def test_constants_match_binding():
    d = _defines()
    for k, v in d.items():
        if hasattr(fa, k):
            assert getattr(fa, k) == v, k
    assert d["FA_KEY_FLAT"] == -1 and d["FA_FLAT_OUT"] == 1 and d["FA_STAGE_HOST"] == 2


def test_strerror_covers_all_codes(lib):
    codes = [v for k, v in _defines().items() if k.startswith("FA_ERR_") or k == "FA_OK"]
    texts = [fa.fa_strerror(c) for c in codes]
    assert all(texts) and len(set(texts)) == len(texts)
    assert fa.fa_strerror(-999) == "unknown status"


def test_argument_errors_need_no_device(lib):
    ctx = ctypes.c_void_p()
    keys = (fa.fa_key * 1)(fa.fa_key(b"w", 4))
    assert lib.fa_open(keys, 1, 0, 0, 1, None, None) == fa.FA_ERR_ARG
    assert lib.fa_open(None, 1, 0, 0, 1, None, ctypes.byref(ctx)) == fa.FA_ERR_ARG
    assert lib.fa_open(keys, 0, 0, 0, 1, None, ctypes.byref(ctx)) == fa.FA_ERR_ARG
    assert lib.fa_open(keys, 1, 0, 0, 0, None, ctypes.byref(ctx)) == fa.FA_ERR_ARG
    assert lib.fa_open(keys, 1, 7, 0, 1, None, ctypes.byref(ctx)) == fa.FA_ERR_DTYPE
    assert lib.fa_open(keys, 1, 0, 2, 1, None, ctypes.byref(ctx)) == fa.FA_ERR_DTYPE
    zero = (fa.fa_key * 1)(fa.fa_key(b"w", 0))
    assert lib.fa_open(zero, 1, 0, 0, 1, None, ctypes.byref(ctx)) == fa.FA_ERR_ARG
    assert ctx.value is None
    assert lib.fa_close(None) == fa.FA_OK
    assert lib.fa_sync(None) == fa.FA_ERR_ARG
    assert lib.fa_reset(None) == fa.FA_ERR_ARG
    assert lib.fa_accumulate(None, 0, 1.0, 0, 0, None, 0, None) == fa.FA_ERR_ARG
    assert lib.fa_accumulate_final(None, 0, 1.0, 0, 0, None, 0, None, None) == fa.FA_ERR_ARG
    assert lib.fa_finalize(None, None, None) == fa.FA_ERR_ARG
    assert lib.fa_finalize_apply(None, None, None, 1.0, None) == fa.FA_ERR_ARG
    assert fa.fa_last_error(None) == ""


def test_binding_checks_batch_lengths(lib):
    """Lists of clients, weights and chunks of different lengths are refused before the
    library is called (ctypes would otherwise pad missing weights with zeros)."""
    with pytest.raises(ValueError, match="lengths differ"):
        fa.fa_accumulate_batch(None, [0, 1], [1.0], 0, 0, [0, 0], 4)
    with pytest.raises(ValueError, match="lengths differ"):
        fa.fa_reduce_resident(None, [0, 1], [1.0, 2.0], [0], [0])
    with pytest.raises(ValueError, match="lengths differ"):
        fa.fa_aggregate_noalloc([1.0, 2.0, 3.0], [0, 0], 4, "f32", "f32", 0)


def test_noalloc_argument_errors_need_no_device(lib):
    w = (ctypes.c_double * 1)(1.0)
    p = (ctypes.c_void_p * 1)(None)
    assert lib.fa_aggregate_noalloc(1, w, p, fa.FA_NOALLOC_MAX_ELEMS + 1, 0, 0, None, None) == fa.FA_ERR_RANGE
    assert lib.fa_aggregate_noalloc(1, w, p, 8, 5, 0, None, None) == fa.FA_ERR_DTYPE
    assert lib.fa_aggregate_noalloc(1, w, p, 8, 0, 0, None, None) == fa.FA_ERR_ARG
    bad = (ctypes.c_double * 1)(float("nan"))
    assert lib.fa_aggregate_noalloc(1, bad, p, 8, 0, 0, 1, None) == fa.FA_ERR_WEIGHT
    assert lib.fa_aggregate_noalloc(0, w, p, 8, 0, 0, None, None) == fa.FA_OK


def test_open_without_a_device_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ctx = ctypes.c_void_p()
    keys = (fa.fa_key * 1)(fa.fa_key(b"w", 4))
    st = lib.fa_open(keys, 1, 0, 0, 1, None, ctypes.byref(ctx))
    assert st in (fa.FA_ERR_CUDA, fa.FA_ERR_NOMEM) and ctx.value is None


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        fa.lib()


def build_c_example():
    """Compile tests/native/abi_example.c -- plain C11 against include/fedavg.h, linked to
    the library and the CUDA runtime -- and return the executable's path."""
    import subprocess
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    out_dir = os.path.join(here, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "abi_example")
    libdir = os.path.dirname(fa.LIB_PATH)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(root, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(here, "native", "abi_example.c"), "-L", libdir, "-lfedavg",
           "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_header_is_c_and_links(lib):
    """The header compiles as plain C11 (warnings as errors) and a C program links against
    the library: the ABI needs neither Python nor C++."""
    assert os.path.exists(build_c_example())
