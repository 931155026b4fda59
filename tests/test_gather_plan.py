"""Host planning of a subset-reduce launch (the round-level adapter reduce): the tiles
of every key written are numbered in order (a key with J reporters in tiles of the most
elements that J reporter tiles fit in one stage) and split into chunks -- contiguous runs
of about equal HBM bytes, each tile of key p moving cnt * (J_p * s_in + s_out) bytes, each
chunk told the key its first tile is in -- which the persistent CTAs take one by one.  Checked against a brute-force walk over every tile
in exact integers, and for the properties the kernel relies on (a monotone split that
starts at tile 0 and ends at the last tile)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "server_side_fedavg_gb300", "csrc")
SO = os.path.join(HERE, "_build", "libplan_shim.so")
CUDA_INC = "/usr/local/cuda/include"

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.isdir(CUDA_INC):
            pytest.skip("CUDA headers are not installed")
        os.makedirs(os.path.dirname(SO), exist_ok=True)
        srcs = [os.path.join(HERE, "native", "plan_shim.cpp"), os.path.join(CSRC, "gather_plan.cpp")]
        deps = srcs + [os.path.join(CSRC, f) for f in ("kernels.cuh", "gather.cuh", "tiles.hpp")]
        if not os.path.exists(SO) or any(os.path.getmtime(s) > os.path.getmtime(SO) for s in deps):
            subprocess.run(["g++", "-O1", "-g", "-std=c++17", "-fPIC", "-shared", "-I", CSRC,
                            "-I", CUDA_INC] + srcs + ["-o", SO], check=True)
        L = ctypes.CDLL(SO)
        vp, u32, i32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32
        L.gp_plan.argtypes = [vp, vp, u32, ctypes.c_int, ctypes.c_int, u32, vp, vp, vp, vp]
        L.gp_plan.restype = i32
        L.gp_chunks.argtypes = [u32, u32]
        L.gp_chunks.restype = u32
        _lib = L
    return _lib


def plan(lens, J, din, dout, grid):
    lens = np.ascontiguousarray(lens, np.uint64)
    J = np.ascontiguousarray(J, np.uint32)
    n = len(lens)
    tiles, ntiles = np.zeros(max(1, n), np.uint32), ctypes.c_uint32()
    tile0 = np.zeros(max(1, n), np.uint32)
    pairs = np.zeros(2 * (grid + 1), np.uint32)
    st = lib().gp_plan(lens.ctypes.data, J.ctypes.data, n, din, dout, grid, tiles.ctypes.data,
                       ctypes.byref(ntiles), tile0.ctypes.data, pairs.ctypes.data)
    assert st == 0
    cta, seg = pairs[0::2], pairs[1::2]
    # the start segment of each CTA: the last segment whose first tile is at or before
    # the CTA's first tile (where the kernel's forward walk over the table begins)
    for f, sg in zip(cta, seg):
        assert sg == max(i for i in range(n) if tile0[i] <= f), (f, sg)
    return tiles[:n], ntiles.value, tile0[:n], cta


STAGE_BYTES = 73728


def tile_for(j, din):
    """Elements per tile of a key with j reporters: the most that j reporter tiles fit in
    one 73,728-byte stage, a multiple of 256."""
    return STAGE_BYTES // (j * (4 if din == 0 else 2)) // 256 * 256


def tile_bytes(lens, J, tiles, din, dout):
    """Bytes of every tile in order (exact integers)."""
    si, so = (4 if din == 0 else 2), (4 if dout == 0 else 2)
    out = []
    for n, j, tile in zip(lens, J, tiles):
        n, tile = int(n), int(tile)
        full, rem = divmod(n, tile)
        out += [tile * (int(j) * si + so)] * full
        if rem:
            out.append(rem * (int(j) * si + so))
    return out


def brute_split(cost, grid):
    """Boundary b = the first tile t whose preceding bytes P(t) satisfy P(t)*grid >= total*b."""
    total = sum(cost)
    prefix = [0]
    for c in cost:
        prefix.append(prefix[-1] + c)
    cta = [0]
    for b in range(1, grid):
        t = next((i for i, p in enumerate(prefix[:-1]) if p * grid >= total * b), len(cost))
        cta.append(t)
    cta.append(len(cost))
    return cta


CASES = [
    # (lens, J, din, dout, grid)
    ([65536] * 16, [8, 4, 6, 7, 5, 8, 8, 4, 5, 6, 7, 8, 4, 4, 6, 5], 1, 1, 152),   # LoRA-like
    ([65536, 65536, 100, 3, 4096 * 3 + 1], [8, 1, 16, 2, 5], 1, 1, 7),
    ([1, 1, 1], [1, 2, 3], 0, 0, 3),
    ([10 ** 6, 17, 10 ** 5], [16, 1, 9], 0, 1, 152),
    ([4096 * 40], [3], 1, 0, 152),
]


@pytest.mark.parametrize("lens,J,din,dout,grid", CASES)
def test_split_matches_the_brute_force_definition(lens, J, din, dout, grid):
    tiles, ntiles, tile0, cta = plan(lens, J, din, dout, grid)
    assert list(tiles) == [tile_for(j, din) for j in J]
    cost = tile_bytes(lens, J, tiles, din, dout)
    assert ntiles == len(cost)
    starts = np.cumsum([0] + [-(-int(n) // int(t)) for n, t in zip(lens, tiles)])[:-1]
    assert list(tile0) == list(starts)
    assert list(cta) == brute_split(cost, grid)


def test_tile_sizes():
    # a stage holds J reporter tiles: bf16 in, J = 8 -> 4608 elements (8 x 9,216 B), J = 1
    # -> 36,864, J = 16 -> 2304; fp32 in, J = 16 -> 1024 (16 x 4,096 B), J = 3 -> 6144
    tiles, _, _, _ = plan([10, 10, 10], [8, 1, 16], 1, 1, 1)
    assert list(tiles) == [4608, 36864, 2304]
    tiles, _, _, _ = plan([10, 10], [16, 3], 0, 0, 1)
    assert list(tiles) == [1024, 6144]
    for j in range(1, 17):
        for din, s in ((0, 4), (1, 2)):
            t = tile_for(j, din)
            assert t % 256 == 0 and j * t * s <= STAGE_BYTES < j * (t + 256) * s


def test_random_rounds_match_and_balance():
    rng = np.random.default_rng(7)
    for _ in range(60):
        n = int(rng.integers(1, 40))
        lens = rng.integers(1, 300000, n)
        small = rng.random(n) < 0.2
        lens[small] = rng.integers(1, 9, int(small.sum()))
        J = rng.integers(1, 17, n)
        din, dout = int(rng.integers(0, 2)), int(rng.integers(0, 2))
        tiles, ntiles, _, _ = plan(lens, J, din, dout, 1)
        grid = int(min(ntiles, rng.integers(1, 400)))
        tiles, ntiles, _, cta = plan(lens, J, din, dout, grid)
        cost = tile_bytes(lens, J, tiles, din, dout)
        assert list(cta) == brute_split(cost, grid)
        assert cta[0] == 0 and cta[-1] == ntiles and np.all(np.diff(cta.astype(np.int64)) >= 0)
        # every CTA's bytes are within one tile of the even share
        total, biggest = sum(cost), max(cost)
        pre = np.concatenate([[0], np.cumsum(cost)])
        per = pre[cta[1:]] - pre[cta[:-1]]
        assert per.max() <= total / grid + biggest


def test_more_ctas_than_bytes_need():
    # a single tile and several CTAs: one CTA takes it, the others take nothing
    tiles, ntiles, _, cta = plan([5], [2], 1, 1, 1)
    assert ntiles == 1 and list(cta) == [0, 1]
    tiles, _, _, cta = plan([5, 7], [2, 3], 1, 1, 2)
    assert list(cta) == brute_split(tile_bytes([5, 7], [2, 3], tiles, 1, 1), 2)


def test_chunk_count():
    f = lib().gp_chunks
    assert f(4096, 152) == 1024          # about four tiles per chunk
    assert f(100, 152) == 100            # never more chunks than tiles
    assert f(300, 152) == 152            # at least one chunk per CTA
    assert f(1 << 30, 152) == 65536      # a bounded table
    for ntiles, grid in ((1, 1), (5, 5), (7, 3), (10 ** 6, 1216)):
        n = f(ntiles, grid)
        assert grid <= n <= ntiles and n <= max(grid, 65536)
