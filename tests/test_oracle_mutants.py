"""The pins have teeth: plausible mistakes planted in a scratch copy of the
oracle source (dropped weight, wrong denominator, global instead of per-key
total, reversed tie rule, off-by-one exponent, dropped last client) are each
caught by the exact-rational and hand-sum pins.  The shipped oracle is never
modified; each mutant is compiled on the CPU into a temporary directory."""
import ctypes
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

from tests import exact

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "fedavg_oracle.c")

MUTANTS = {
    "dropped_weight": ("if (reported[k]) s += n[k] * fo_load(x[k], dtype_in, i);",
                       "if (reported[k]) s += fo_load(x[k], dtype_in, i);"),
    "count_denominator": ("double y = s / N;\n        if (dtype_out", "double y = s / (double)cnt;\n        if (dtype_out"),
    "ignores_mask": ("if (reported[k]) s += n[k]", "s += n[k]"),
    "last_client_dropped": ("for (uint32_t k = 0; k < K; ++k) {\n            if (reported[k]) s +=",
                            "for (uint32_t k = 0; k + 1 < K; ++k) {\n            if (reported[k]) s +="),
    "ties_away": ("else k = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "else k = fl + 1.0;"),
    "wrong_quantum": ("double q = ldexp(1.0, E - 7);", "double q = ldexp(1.0, E - 8);"),
    "truncating_cast": ("if (frac > 0.5) k = fl + 1.0;", "if (frac > 2.0) k = fl + 1.0;"),
}

APPLY_MUTANTS = {
    "apply_drops_base": ("double y = fo_load(base, dtype_out, i) + server_lr * (s / N);",
                         "double y = server_lr * (s / N);"),
    "apply_drops_lr": ("double y = fo_load(base, dtype_out, i) + server_lr * (s / N);",
                       "double y = fo_load(base, dtype_out, i) + (s / N);"),
    "apply_sign": ("double y = fo_load(base, dtype_out, i) + server_lr * (s / N);",
                   "double y = fo_load(base, dtype_out, i) - server_lr * (s / N);"),
}


def _build(tmp, name, a, b):
    src = open(SRC).read()
    assert a in src, f"mutation anchor for {name} not found"
    mutated = src.replace(a, b, 1)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"{name}.so")
    open(c, "w").write(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", c, "-o", so, "-lm"],
                   check=True)
    L = ctypes.CDLL(so)
    u32, u64, i32, f64, vp = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    L.fo_fedavg_key.argtypes = [u32, vp, vp, vp, i32, u64, i32, vp, vp, vp]
    L.fo_fedavg_key.restype = i32
    L.fo_fedavg_apply_key.argtypes = [u32, vp, vp, vp, i32, u64, vp, f64, i32, vp, vp, vp]
    L.fo_fedavg_apply_key.restype = i32
    return L


def _run_key(L, weights, reported, xs, code_in, code_out):
    K = len(weights)
    n = np.asarray(weights, np.float64)
    rep = np.asarray(reported, np.uint8)
    m = next(x.size for x, r in zip(xs, reported) if r)
    ptrs = (ctypes.c_void_p * K)(*[x.ctypes.data for x in xs])
    out = np.zeros(m, np.float32 if code_out == 0 else np.uint16)
    L.fo_fedavg_key(K, n.ctypes.data, rep.ctypes.data, ptrs, code_in, m, code_out, out.ctypes.data, None, None)
    return out


def _pins_pass(L) -> bool:
    """A compact replay of the exact-rational pin (bf16 and fp32 outputs)."""
    rng = np.random.default_rng(99)
    for trial in range(30):
        K = int(rng.integers(2, 6))
        m = 16
        weights = [float(v) for v in rng.integers(1, 5000, K)]
        reported = [True] * K
        if trial % 3 == 0:
            reported[0] = False
        xs = [(rng.standard_normal(m) * 10.0 ** rng.uniform(-3, 1)).astype(np.float32) for _ in range(K)]
        ex = exact.exact_fedavg(weights, reported, [x.astype(np.float64).tolist() for x in xs])
        got32 = _run_key(L, weights, reported, xs, 0, 0)
        if got32.view(np.uint32).tolist() != [exact.nearest_f32(v) for v in ex]:
            return False
        got16 = _run_key(L, weights, reported, xs, 0, 1)
        if got16.tolist() != [exact.nearest_bf16(v) for v in ex]:
            return False
        # exact bf16 ties: y = midpoint between two bf16 neighbours
        b = int(rng.integers(0x3000, 0x4000))
        mid = float((exact.bf16_bits_to_fraction(b) + exact.bf16_bits_to_fraction(b + 1)) / 2)
        x = np.array([mid], np.float32)
        got = _run_key(L, [3.0], [True], [x], 0, 1)
        if got.tolist() != [exact.nearest_bf16(Fraction(mid))]:
            return False
    return True


def _apply_pins_pass(L) -> bool:
    """A compact replay of the delta-round exact-rational pin."""
    rng = np.random.default_rng(98)
    for trial in range(20):
        K, m = int(rng.integers(1, 5)), 8
        weights = [float(v) for v in rng.integers(1, 3000, K)]
        xs = [(rng.standard_normal(m) * 1e-3).astype(np.float32) for _ in range(K)]
        base = (rng.standard_normal(m) * 0.02).astype(np.float32)
        lr = float(rng.choice([0.5, 2.0]))
        ptrs = (ctypes.c_void_p * K)(*[x.ctypes.data for x in xs])
        n = np.asarray(weights, np.float64)
        rep = np.ones(K, np.uint8)
        out = np.zeros(m, np.float32)
        L.fo_fedavg_apply_key(K, n.ctypes.data, rep.ctypes.data, ptrs, 0, m, base.ctypes.data, lr, 0,
                              out.ctypes.data, None, None)
        mean = exact.exact_fedavg(weights, [True] * K, [x.astype(np.float64).tolist() for x in xs])
        want = [exact.nearest_f32(Fraction(float(base[i])) + Fraction(lr) * mean[i]) for i in range(m)]
        if out.view(np.uint32).tolist() != want:
            return False
    return True


def test_unmutated_copy_passes(tmp_path):
    src = open(SRC).read()
    L = _build(str(tmp_path), "identity", src[:10], src[:10])
    assert _pins_pass(L)
    assert _apply_pins_pass(L)


@pytest.mark.parametrize("name", sorted(APPLY_MUTANTS))
def test_apply_mutant_is_caught(tmp_path, name):
    a, b = APPLY_MUTANTS[name]
    L = _build(str(tmp_path), name, a, b)
    assert not _apply_pins_pass(L), f"pins did not catch mutant {name}"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    a, b = MUTANTS[name]
    L = _build(str(tmp_path), name, a, b)
    assert not _pins_pass(L), f"pins did not catch mutant {name}"
