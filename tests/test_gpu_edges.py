"""GPU edge cases and error behaviour through the C ABI."""
import threading

import numpy as np
import pytest
import torch

import oracle
import synth
import server_side_fedavg_gb300 as fa
from tests.compare import Bf16Tally, check_bf16, check_f32, check_f32_to_bf16, fp32_sum_model
from tests.gpu_helpers import sentinel, sentinel_np, to_dev, to_np, to_pinned

pytestmark = pytest.mark.gpu


def _bf16(rng, n, s=0.05):
    return ((rng.standard_normal(n) * s).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _f32(rng, n, s=0.05):
    return (rng.standard_normal(n) * s).astype(np.float32)


@pytest.mark.parametrize("din,dout", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16")])
def test_odd_sizes_and_misaligned_chunks(din, dout):
    """numel 1 / 7 / 4097 / 3 tiles + 5, chunks at odd offsets (unaligned pointers:
    scalar path) and whole (vector path); unreported and zero-weight keys untouched."""
    rng = np.random.default_rng(1)
    numels = [1, 7, 4097, 3 * 4096 + 5, 33, 100]
    K = 4
    weights = [300.0, 0.0, 1000.0, 17.0]
    gen = _f32 if din == "f32" else _bf16
    xs = [[gen(rng, n) for n in numels] for _ in range(K)]
    # key 4: nobody; key 5: only client 1 (weight 0)
    reports = [[p for p in range(len(numels)) if p not in (4, 5)] for _ in range(K)]
    reports[1] = reports[1] + [5]
    ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], din, dout, K)
    tally = Bf16Tally()
    try:
        for k in range(K):
            for p in reports[k]:
                t = to_dev(xs[k][p])
                n = numels[p]
                es = t.element_size()
                cuts = [0, min(3, n), min(n, 3 + 4099), n] if k % 2 else [0, n]
                for a, b in zip(cuts[:-1], cuts[1:]):
                    if b > a:
                        fa.fa_accumulate(ctx, k, weights[k], p, a, t.data_ptr() + a * es, b - a)
                fa.fa_accumulate(ctx, k, weights[k], p, 0, t.data_ptr(), 0)   # empty chunk: no-op
        outs = [sentinel(n, dout) for n in numels]
        fa.fa_finalize(ctx, outs)
        torch.cuda.synchronize()
        for p, n in enumerate(numels):
            rep = [p in reports[k] for k in range(K)]
            want, N, cnt = oracle.fedavg_key(weights, rep, [xs[k][p] for k in range(K)], din, dout)
            got = to_np(outs[p], dout)
            assert fa.fa_key_total(ctx, p) == (N, cnt)
            if want is None:
                assert np.array_equal(got, sentinel_np(n, dout)), f"key {p} was written"
            else:
                mx = max(float(np.abs(xs[k][p].astype(np.float64) if din == "f32" else
                                      (xs[k][p].astype(np.uint32) << 16).view(np.float32)).max())
                         for k in range(K) if rep[k])
                if dout == "f32":
                    check_f32(got, want, mx, cnt, f"key {p}")
                elif din == "f32":
                    check_f32_to_bf16(got, want, mx, cnt, f"key {p}")
                else:
                    tally.add(got, want, f"key {p}")
        if dout == "bf16" and din == "bf16":
            tally.check(f"{din}->{dout}")
    finally:
        fa.fa_close(ctx)


def test_single_client_and_identical_clients_bit_exact():
    rng = np.random.default_rng(2)
    x = _bf16(rng, 10000, 0.02)
    for K in (1, 5):
        ctx = fa.fa_open([("w", x.size)], "bf16", "bf16", K)
        try:
            t = to_dev(x)
            for k in range(K):
                fa.fa_accumulate(ctx, k, float(100 + 37 * k), 0, 0, t, x.size)
            out = sentinel(x.size, "bf16")
            fa.fa_finalize(ctx, [out])
            torch.cuda.synchronize()
            assert np.array_equal(to_np(out, "bf16"), x)
        finally:
            fa.fa_close(ctx)


def test_finalize_twice_and_rounds():
    rng = np.random.default_rng(3)
    n = 5000
    a, b = _f32(rng, n), _f32(rng, n)
    ctx = fa.fa_open([("w", n)], "f32", "f32", 2)
    try:
        ta, tb = to_dev(a), to_dev(b)
        fa.fa_accumulate(ctx, 0, 3.0, 0, 0, ta, n)
        fa.fa_accumulate(ctx, 1, 1.0, 0, 0, tb, n)
        o1, o2 = sentinel(n, "f32"), sentinel(n, "f32")
        fa.fa_finalize(ctx, [o1])
        fa.fa_finalize(ctx, [o2])
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_accumulate(ctx, 0, 3.0, 0, 0, ta, n)
        assert e.value.status == fa.FA_ERR_STATE
        fa.fa_reset(ctx)
        # next round: only client 1, new weight (a power of two: 8*b/8 == b exactly)
        fa.fa_accumulate(ctx, 1, 8.0, 0, 0, tb, n)
        o3 = sentinel(n, "f32")
        fa.fa_finalize(ctx, [o3])
        torch.cuda.synchronize()
        assert np.array_equal(o3.cpu().numpy(), b)
        assert fa.fa_key_total(ctx, 0) == (8.0, 1)
    finally:
        fa.fa_close(ctx)


def test_error_codes():
    n = 100
    x = to_dev(np.zeros(n, np.float32))
    ctx = fa.fa_open([("a", n), ("b", 10)], "f32", "bf16", 2)
    try:
        def code(f, *a):
            with pytest.raises(fa.FedAvgError) as e:
                f(*a)
            return e.value.status
        assert code(fa.fa_accumulate, ctx, 2, 1.0, 0, 0, x, n) == fa.FA_ERR_ARG           # client id
        assert code(fa.fa_accumulate, ctx, 0, 1.0, 2, 0, x, 1) == fa.FA_ERR_ARG           # key id
        assert code(fa.fa_accumulate, ctx, 0, 1.0, 0, 1, x, n) == fa.FA_ERR_RANGE         # past the key
        assert code(fa.fa_accumulate, ctx, 0, 1.0, -1, 105, x, 6) == fa.FA_ERR_RANGE      # past flat end
        assert code(fa.fa_accumulate, ctx, 0, -1.0, 0, 0, x, n) == fa.FA_ERR_WEIGHT
        assert code(fa.fa_accumulate, ctx, 0, float("nan"), 0, 0, x, n) == fa.FA_ERR_WEIGHT
        assert code(fa.fa_accumulate, ctx, 0, 2.0 ** 24 + 1, 0, 0, x, n) == fa.FA_ERR_WEIGHT
        fa.fa_accumulate(ctx, 0, 5.0, 0, 0, x, 50)
        assert code(fa.fa_accumulate, ctx, 0, 6.0, 0, 50, x, 50) == fa.FA_ERR_WEIGHT      # weight changed
        assert code(fa.fa_accumulate, ctx, 0, 5.0, 0, 20, x, 51) == fa.FA_ERR_RANGE       # over-coverage
        host = np.zeros(n, np.float32)
        assert code(fa.fa_accumulate_batch, ctx, [1, 0], [1.0, 5.0], 0, 0, [host, x], n) == fa.FA_ERR_ARG   # mix
        assert code(fa.fa_accumulate_batch, ctx, [1, 1], [1.0, 1.0], 0, 0, [x, x], n) == fa.FA_ERR_ARG
        out = [torch.empty(n, dtype=torch.int16, device="cuda"), torch.empty(10, dtype=torch.int16, device="cuda")]
        assert code(fa.fa_finalize, ctx, out) == fa.FA_ERR_INCOMPLETE                      # client 0 sent half
        fa.fa_accumulate(ctx, 0, 5.0, 0, 50, x.data_ptr() + 200, 50)
        fa.fa_finalize(ctx, out)
        assert fa.fa_get_stats(ctx)["chunks"] == 2
    finally:
        fa.fa_close(ctx)


def _classes(v):
    """0 finite, 1 NaN, 2 +inf, 3 -inf."""
    return np.where(np.isnan(v), 1, np.where(v == np.inf, 2, np.where(v == -np.inf, 3, 0)))


@pytest.mark.parametrize("din,dout", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("mode", ["device", "pinned"])
def test_non_finite_values_propagate_as_ieee(din, dout, mode):
    """No special cases for non-finite inputs (IEEE propagation): +inf and -inf pass
    through, inf + (-inf) and NaN give NaN, and a zero-weight client's inf gives NaN
    (0 * inf) -- as the fp64 oracle computes; finite elements keep their bounds."""
    rng = np.random.default_rng(21)
    n = 3 * 4096 + 7
    K = 3
    w = [3.0, 5.0, 0.0]
    xs = [(_f32(rng, n) if din == "f32" else _bf16(rng, n)) for _ in range(K)]
    if din == "f32":
        pinf, ninf, nan = np.float32(np.inf), np.float32(-np.inf), np.float32(np.nan)
    else:
        pinf, ninf, nan = np.uint16(0x7F80), np.uint16(0xFF80), np.uint16(0x7FC0)
    plant = {(0, 10): pinf, (1, 20): nan, (0, 30): pinf, (1, 30): ninf, (2, 40): pinf,
             (0, 50): ninf, (0, 4100): nan, (1, n - 1): pinf}
    for (k, i), v in plant.items():
        xs[k][i] = v
    ctx = fa.fa_open([("k", n)], din, dout, K)
    try:
        keep = []
        for k in range(K):
            t = to_dev(xs[k]) if mode == "device" else to_pinned(xs[k])
            keep.append(t)
            fa.fa_accumulate(ctx, k, w[k], 0, 0, t, n)
        out = sentinel(n, dout)
        fa.fa_finalize(ctx, [out])
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
    finally:
        fa.fa_close(ctx)
    got = to_np(out, dout)
    want, _, _ = oracle.fedavg_key(w, [True] * K, xs, din, dout)
    as_f = (lambda b: (b.astype(np.uint32) << 16).view(np.float32)) if dout == "bf16" else (lambda a: a)
    g, wv = as_f(got), as_f(want)
    assert np.array_equal(_classes(g), _classes(wv))
    expect_bad = {10: 2, 20: 1, 30: 1, 40: 1, 50: 3, 4100: 1, n - 1: 2}
    for i, c in expect_bad.items():
        assert _classes(wv[i:i + 1])[0] == c, i
    fin = _classes(wv) == 0
    mx = max(float(np.abs(np.nan_to_num((xs[k].astype(np.uint32) << 16).view(np.float32)
                                         if din == "bf16" else xs[k], posinf=0, neginf=0)).max())
             for k in range(K))
    if dout == "f32":
        check_f32(got[fin], want[fin], mx, K, "finite elements")
    else:
        check_f32_to_bf16(got[fin], want[fin], mx, K, "finite elements")


def test_host_outputs_match_device_outputs():
    """Pinned outputs written in place by the kernel or staged through a device buffer
    (FA_STAGE_HOST), pageable outputs (always staged), per key or flat (flat keys start
    unaligned): the same bits as device outputs, and the bytes sent to the host are
    counted."""
    rng = np.random.default_rng(4)
    numels = [4096 * 2 + 3, 9, 70000]
    K = 3
    xs = [[_bf16(rng, n) for n in numels] for _ in range(K)]
    w = [10.0, 20.0, 30.0]
    res = {}
    modes = ("device", "pinned", "pinned_staged", "pageable", "pageable_staged", "flat_pinned",
             "flat_pinned_staged", "flat_pageable")
    for mode in modes:
        flags = (fa.FA_FLAT_OUT if mode.startswith("flat") else 0) | \
                (fa.FA_STAGE_HOST if mode.endswith("staged") else 0)
        ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], "bf16", "bf16", K, flags=flags)
        try:
            for k in range(K):
                for p in (0, 2):                      # key 1 never sent: must stay untouched
                    fa.fa_accumulate(ctx, k, w[k], p, 0, to_dev(xs[k][p]), numels[p])
            if mode == "device":
                outs = [sentinel(n, "bf16") for n in numels]
            elif mode.startswith("pinned"):
                outs = [sentinel(n, "bf16", "cpu").pin_memory() for n in numels]
            elif mode.startswith("pageable"):
                outs = [sentinel_np(n, "bf16").copy() for n in numels]
            elif mode == "flat_pageable":
                outs = [sentinel_np(sum(numels), "bf16").copy()]
            else:
                outs = [sentinel(sum(numels), "bf16", "cpu").pin_memory()]
            fa.fa_finalize(ctx, outs)
            fa.fa_sync(ctx)
            torch.cuda.synchronize()
            sent = fa.fa_get_stats(ctx)["d2h_bytes"]
            assert sent == (0 if mode == "device" else 2 * (numels[0] + numels[2])), (mode, sent)
            got = [to_np(o, "bf16") if isinstance(o, torch.Tensor) else o for o in outs]
            if mode.startswith("flat"):
                offs = np.cumsum([0] + numels)
                got = [got[0][offs[i]:offs[i + 1]] for i in range(len(numels))]
            res[mode] = got
        finally:
            fa.fa_close(ctx)
    for mode in res:
        for p in range(len(numels)):
            assert np.array_equal(res[mode][p], res["device"][p]), (mode, p)
    assert np.array_equal(res["device"][1], sentinel_np(numels[1], "bf16"))


@pytest.mark.parametrize("staged", [False, True])
def test_pageable_chunk_reusable_on_return(staged):
    """A pageable chunk has been consumed when fa_accumulate returns (read in place and
    waited for, or copied into staging): overwriting it at once changes nothing."""
    rng = np.random.default_rng(12)
    n = 3 * 4096 * 8 + 5
    xs = [_bf16(rng, n) for _ in range(3)]
    w = [3.0, 5.0, 7.0]
    flags = fa.FA_STAGE_HOST if staged else 0
    ctx = fa.fa_open([("k", n)], "bf16", "bf16", 3, flags=flags, ring_slots=2, slot_bytes=1 << 16)
    try:
        s = torch.cuda.Stream()
        buf = np.empty(n, np.uint16)
        for k in range(3):
            buf[:] = xs[k]
            fa.fa_accumulate(ctx, k, w[k], 0, 0, buf, n, s)
            buf[:] = 0x7FC0                            # NaN bits: must not reach the sum
        out = sentinel(n, "bf16")
        fa.fa_finalize(ctx, [out], s)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        want, _, _ = oracle.fedavg_key(w, [True] * 3, xs, "bf16", "bf16")
        check_bf16(to_np(out, "bf16"), want, "pageable reuse")
    finally:
        fa.fa_close(ctx)


def test_bounded_wait_times_out_then_recovers():
    """fa_sync returns FA_ERR_TIMEOUT (never hangs) while queued work is still
    running, here a bounded sleep kernel queued ahead of the accumulate."""
    n = 1 << 16
    x = to_dev(np.ones(n, np.float32))
    ctx = fa.fa_open([("w", n)], "f32", "f32", 1, timeout_ms=5)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            torch.cuda._sleep(500_000_000)        # ~0.25 s of spinning, then it ends
        fa.fa_accumulate(ctx, 0, 2.0, 0, 0, x, n, s)
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_sync(ctx)
        assert e.value.status == fa.FA_ERR_TIMEOUT
        s.synchronize()
        fa.fa_sync(ctx)
        out = torch.empty(n, dtype=torch.float32, device="cuda")
        fa.fa_finalize(ctx, [out], s)
        s.synchronize()
        assert bool((out == 1.0).all())
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_concurrent_client_threads():
    """Clients arriving on several host threads and streams; order varies, the
    result stays within tolerance of the oracle and the totals are exact."""
    rng = np.random.default_rng(6)
    numels = [4096 * 5 + 1, 1000, 123457]
    K = 8
    xs = [[_f32(rng, n, 0.02) for n in numels] for _ in range(K)]
    w = [float(v) for v in rng.integers(100, 1001, K)]
    ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], "f32", "f32", K)
    errors = []
    dx = [[to_dev(xs[k][p]) for p in range(len(numels))] for k in range(K)]
    torch.cuda.synchronize()

    def client(k):
        try:
            s = torch.cuda.Stream()
            for p, n in enumerate(numels):
                fa.fa_accumulate(ctx, k, w[k], p, 0, dx[k][p], n, s)
            s.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    try:
        th = [threading.Thread(target=client, args=(k,)) for k in range(K)]
        for t in th:
            t.start()
        for t in th:
            t.join()
        assert not errors, errors
        outs = [torch.empty(n, dtype=torch.float32, device="cuda") for n in numels]
        fa.fa_finalize(ctx, outs)
        torch.cuda.synchronize()
        for p, n in enumerate(numels):
            want, N, cnt = oracle.fedavg_key(w, [True] * K, [xs[k][p] for k in range(K)], "f32", "f32")
            mx = max(float(np.abs(xs[k][p]).max()) for k in range(K))
            check_f32(outs[p].cpu().numpy(), want, mx, K, f"key {p}")
            assert fa.fa_key_total(ctx, p) == (N, cnt)
    finally:
        fa.fa_close(ctx)


@pytest.mark.slow
@pytest.mark.parametrize("dout", ["bf16", "f32"])
def test_key_of_more_than_2_pow_32_elements(dout):
    """One key of 2^32 + 77 bf16 elements, so offsets inside a single segment pass 2^31 and
    2^32: two clients streamed whole, then the same two reduced resident (fa_reduce_resident),
    sampled against the oracle around 2^31, 2^32 and the ragged end; bf16 and fp32 output."""
    n = (1 << 32) + 77
    so = 2 if dout == "bf16" else 4
    need = 2 * n * 2 + n * 4 + n * so + (4 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.fail(f"needs {need / 1e9:.0f} GB free, have {free / 1e9:.0f}")
    seed, sigma = 4242, 0.02
    w = [700.0, 300.0]
    s = torch.cuda.current_stream()
    xd = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(2)]
    for k in range(2):
        synth.fill_device(seed, k, 0, sigma, "bf16", 0, n, xd[k].data_ptr(), s.cuda_stream)
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([
        np.arange(0, 64), np.arange((1 << 31) - 64, (1 << 31) + 64),
        np.arange((1 << 32) - 64, (1 << 32) + 64), np.arange(n - 200, n),
        rng.integers(0, n, 20000)])).astype(np.int64)
    tidx = torch.from_numpy(idx).cuda()
    odt = torch.int16 if dout == "bf16" else torch.float32
    out = torch.empty(n, dtype=odt, device="cuda")
    got = {}
    ctx = fa.fa_open([("big", n)], "bf16", dout, 2)
    try:
        for k in range(2):
            fa.fa_accumulate(ctx, k, w[k], 0, 0, xd[k], n, s)
        fa.fa_finalize(ctx, [out], s)
        fa.fa_sync(ctx)
        got["streamed"] = to_np(out[tidx], dout)
    finally:
        fa.fa_close(ctx)
    out.fill_(0x7FBF if dout == "bf16" else -7.0)
    ctx = fa.fa_open([("big", n)], "bf16", dout, 2)
    try:
        fa.fa_reduce_resident(ctx, [0, 1], w, xd, [out], s)
        fa.fa_sync(ctx)
        got["resident"] = to_np(out[tidx], dout)
    finally:
        fa.fa_close(ctx)
    del xd, out
    torch.cuda.empty_cache()
    xs = [synth.gather(seed, k, 0, sigma, "bf16", idx.astype(np.uint64)) for k in range(2)]
    want, N, cnt = oracle.fedavg_key(w, [True, True], xs, "bf16", dout)
    assert (N, cnt) == (1000.0, 2)
    mx = max(float(np.abs(synth.to_f64(x, "bf16")).max()) for x in xs)
    for how, g in got.items():
        if dout == "f32":
            check_f32(g, want, mx, 2, f"2^32 + 77 elements, {how}")
        else:
            check_bf16(g, want, f"2^32 + 77 elements, {how}",
                       model=fp32_sum_model(w, [True, True], xs, "bf16"), bound=1e-6 * mx * 2)
    assert np.array_equal(got["streamed"], got["resident"])


def test_caller_registered_host_memory():
    """Host memory the caller page-locked with cudaHostRegister (a NumPy buffer, say) is
    pinned memory to the library: read in place where the device maps it at the same
    address, else staged.  Same bits as device ingest, ragged chunks included."""
    rng = np.random.default_rng(33)
    n = 5 * 4096 + 13
    K = 3
    xs = [_bf16(rng, n) for _ in range(K)]
    w = [11.0, 13.0, 17.0]
    cudart = torch.cuda.cudart()
    bufs = [np.empty(n + 64, np.uint16) for _ in range(K)]     # registered as a whole
    for b in bufs:
        assert int(cudart.cudaHostRegister(b.ctypes.data, b.nbytes, 0)) == 0
    outs = {}
    try:
        for how in ("registered", "device"):
            ctx = fa.fa_open([("k", n)], "bf16", "bf16", K)
            try:
                keep = []
                for k in range(K):
                    if how == "registered":
                        bufs[k][3:3 + n] = xs[k]                # an odd start inside the region
                        base = bufs[k].ctypes.data + 6
                    else:
                        t = to_dev(xs[k])
                        keep.append(t)
                        base = t.data_ptr()
                    for a, b in [(0, 4097), (4097, 4100), (4100, n)]:
                        fa.fa_accumulate(ctx, k, w[k], 0, a, base + 2 * a, b - a)
                out = sentinel(n, "bf16")
                fa.fa_finalize(ctx, [out])
                fa.fa_sync(ctx)
                torch.cuda.synchronize()
                outs[how] = to_np(out, "bf16")
            finally:
                fa.fa_close(ctx)
    finally:
        torch.cuda.synchronize()
        for b in bufs:
            cudart.cudaHostUnregister(b.ctypes.data)
    assert np.array_equal(outs["registered"], outs["device"])
    want, _, _ = oracle.fedavg_key(w, [True] * K, xs, "bf16", "bf16")
    check_bf16(outs["device"], want, "registered host memory")


def test_fa_log_reports_failures_on_stderr():
    """FA_LOG=1 writes each reported failure to stderr; unset, the library prints nothing."""
    import os
    import subprocess
    import sys
    code = (
        "import numpy as np, server_side_fedavg_gb300 as fa, torch\n"
        "ctx = fa.fa_open([('k', 8)], 'f32', 'f32', 1)\n"
        "x = torch.zeros(8, device='cuda')\n"
        "fa.fa_accumulate(ctx, 0, 2.0, 0, 0, x, 4)\n"
        "try:\n"
        "    fa.fa_accumulate(ctx, 0, 3.0, 0, 4, x, 4)\n"
        "except fa.FedAvgError:\n"
        "    pass\n"
        "fa.fa_close(ctx)\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root)
    for value, expect in (("1", True), (None, False)):
        e = dict(env)
        e.pop("FA_LOG", None)
        if value is not None:
            e["FA_LOG"] = value
        r = subprocess.run([sys.executable, "-c", code], cwd=root, env=e, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        logged = "[fedavg]" in r.stderr and "weight differs" in r.stderr
        assert logged == expect, r.stderr[-2000:]


@pytest.mark.parametrize("kind", ["pinned", "pageable"])
def test_batch_from_host_memory_in_place(kind):
    """fa_accumulate_batch over host chunks the device addresses: one in-place launch per
    client, bit-identical to the same batch from device memory; a device/host mix and host
    chunks under FA_STAGE_HOST are refused with nothing recorded."""
    rng = np.random.default_rng(41)
    n = 3 * 4096 + 11
    J = 5
    xs = [_bf16(rng, n) for _ in range(J)]
    w = [float(v) for v in rng.integers(100, 1001, J)]
    res = {}
    for how in ("device", kind):
        ctx = fa.fa_open([("k", n)], "bf16", "bf16", J)
        try:
            if how == "device":
                ptrs = [to_dev(x) for x in xs]
            elif how == "pinned":
                ptrs = [to_pinned(x) for x in xs]
            else:
                ptrs = [x.copy() for x in xs]
            s = torch.cuda.Stream()
            try:
                fa.fa_accumulate_batch(ctx, list(range(J)), w, 0, 0, ptrs, n, s)
            except fa.FedAvgError as e:
                if how == "pageable" and e.status == fa.FA_ERR_ARG:
                    pytest.skip("this device does not read pageable host memory in place")
                raise
            out = sentinel(n, "bf16")
            fa.fa_finalize(ctx, [out], s)
            fa.fa_sync(ctx)
            torch.cuda.synchronize()
            res[how] = to_np(out, "bf16")
            st = fa.fa_get_stats(ctx)
            assert st["h2d_bytes"] == (0 if how == "device" else J * n * 2)
        finally:
            fa.fa_close(ctx)
    assert np.array_equal(res[kind], res["device"])
    want, _, _ = oracle.fedavg_key(w, [True] * J, xs, "bf16", "bf16")
    check_bf16(res["device"], want, "batch")
    ctx = fa.fa_open([("k", n)], "bf16", "bf16", J)
    try:
        mixed = [to_dev(xs[0]), to_pinned(xs[1])]
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_accumulate_batch(ctx, [0, 1], w[:2], 0, 0, mixed, n)
        assert e.value.status == fa.FA_ERR_ARG and fa.fa_key_total(ctx, 0) == (0.0, 0)
    finally:
        fa.fa_close(ctx)
    ctx = fa.fa_open([("k", n)], "bf16", "bf16", J, flags=fa.FA_STAGE_HOST)
    try:
        with pytest.raises(fa.FedAvgError) as e:
            fa.fa_accumulate_batch(ctx, [0, 1], w[:2], 0, 0, [to_pinned(xs[0]), to_pinned(xs[1])], n)
        assert e.value.status == fa.FA_ERR_ARG
    finally:
        torch.cuda.synchronize()
        fa.fa_close(ctx)


def test_two_contexts_from_two_threads():
    """Two independent aggregations (different layouts and dtypes) driven at once from two
    host threads on one GPU: each matches the oracle; neither sees the other's state."""
    import threading
    rng = np.random.default_rng(55)
    jobs = {
        "a": ([4096 * 7 + 3, 100, 9000], "bf16", "bf16", 4),
        "b": ([70000, 1, 4100], "f32", "f32", 3),
    }
    data, results, errors = {}, {}, []
    for name, (numels, din, dout, K) in jobs.items():
        xs = [[(_bf16(rng, n) if din == "bf16" else _f32(rng, n)) for n in numels] for _ in range(K)]
        w = [float(v) for v in rng.integers(100, 1001, K)]
        data[name] = (xs, w)

    def run(name):
        try:
            numels, din, dout, K = jobs[name]
            xs, w = data[name]
            ctx = fa.fa_open([(f"{name}{i}", n) for i, n in enumerate(numels)], din, dout, K)
            try:
                s = torch.cuda.Stream()
                for rnd in range(3):
                    fa.fa_reset(ctx)
                    keep = []
                    for k in range(K):
                        for p, n in enumerate(numels):
                            t = to_dev(xs[k][p])
                            keep.append(t)
                            fa.fa_accumulate(ctx, k, w[k], p, 0, t, n, s)
                    outs = [sentinel(n, dout) for n in numels]
                    fa.fa_finalize(ctx, outs, s)
                    fa.fa_sync(ctx)
                    s.synchronize()
                results[name] = [to_np(o, dout) for o in outs]
            finally:
                fa.fa_close(ctx)
        except Exception as e:  # reported below
            errors.append(e)

    th = [threading.Thread(target=run, args=(name,)) for name in jobs]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    for name, (numels, din, dout, K) in jobs.items():
        xs, w = data[name]
        for p in range(len(numels)):
            col = [xs[k][p] for k in range(K)]
            want, _, _ = oracle.fedavg_key(w, [True] * K, col, din, dout)
            if dout == "f32":
                check_f32(results[name][p], want, max(float(np.abs(x).max()) for x in col), K, f"{name} {p}")
            else:
                check_bf16(results[name][p], want, f"{name} {p}")


def _managed(n, dtype):
    """n elements of cudaMallocManaged memory (as a NumPy view for the host) and a freer."""
    import ctypes
    fa.lib()                                          # loads the runtime the library links
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaMallocManaged.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
    rt.cudaFree.argtypes = [ctypes.c_void_p]
    p = ctypes.c_void_p()
    itemsize = np.dtype(dtype).itemsize
    assert rt.cudaMallocManaged(ctypes.byref(p), n * itemsize, 1) == 0   # cudaMemAttachGlobal
    view = np.ctypeslib.as_array((ctypes.c_uint8 * (n * itemsize)).from_address(p.value)).view(dtype)
    return p.value, view, lambda: rt.cudaFree(p.value)


def test_managed_memory_inputs_and_outputs():
    """cudaMallocManaged chunks are read in place with plain loads (single calls, a batch,
    a multi-chunk call) and a managed output is written by the finalize kernel: the same
    bits as device memory.  The resident round and delta-apply bases refuse managed memory."""
    rng = np.random.default_rng(61)
    n = 2 * 4096 + 9
    K = 4
    xs = [_bf16(rng, n) for _ in range(K)]
    w = [float(v) for v in rng.integers(100, 1001, K)]
    frees = []
    try:
        mptr = []
        for x in xs:
            p, view, free = _managed(n, np.uint16)
            view[:] = x
            mptr.append(p)
            frees.append(free)
        out_p, out_view, free = _managed(n, np.uint16)
        frees.append(free)
        res = {}
        for how in ("device", "managed"):
            ctx = fa.fa_open([("k", n)], "bf16", "bf16", K)
            try:
                ptrs = [to_dev(x) for x in xs] if how == "device" else mptr
                fa.fa_accumulate(ctx, 0, w[0], 0, 0, ptrs[0], n)                      # single
                fa.fa_accumulate_batch(ctx, [1, 2], w[1:3], 0, 0, ptrs[1:3], n)        # batch
                p3 = ptrs[3] if isinstance(ptrs[3], int) else ptrs[3].data_ptr()
                fa.fa_accumulate_keys(ctx, 3, w[3], [0, 0], [0, 5000], [p3, p3 + 2 * 5000],
                                      [5000, n - 5000])                               # keys
                if how == "device":
                    out = sentinel(n, "bf16")
                    fa.fa_finalize(ctx, [out])
                    fa.fa_sync(ctx)
                    torch.cuda.synchronize()
                    res[how] = to_np(out, "bf16")
                else:
                    out_view[:] = 0x7FBF
                    fa.fa_finalize(ctx, [out_p])
                    fa.fa_sync(ctx)
                    torch.cuda.synchronize()
                    res[how] = out_view.copy()
                    assert fa.fa_get_stats(ctx)["h2d_bytes"] == 0 and fa.fa_get_stats(ctx)["d2h_bytes"] == 0
            finally:
                fa.fa_close(ctx)
        assert np.array_equal(res["managed"], res["device"])
        want, _, _ = oracle.fedavg_key(w, [True] * K, xs, "bf16", "bf16")
        check_bf16(res["device"], want, "managed")
        ctx = fa.fa_open([("k", n)], "bf16", "bf16", K)
        try:
            with pytest.raises(fa.FedAvgError) as e:
                fa.fa_reduce_resident(ctx, list(range(K)), w, mptr, [to_dev(xs[0])])
            assert e.value.status == fa.FA_ERR_ARG
        finally:
            fa.fa_close(ctx)
        ctx = fa.fa_open([("k", n)], "bf16", "bf16", K)
        try:
            fa.fa_accumulate(ctx, 0, w[0], 0, 0, to_dev(xs[0]), n)
            with pytest.raises(fa.FedAvgError) as e:
                fa.fa_finalize_apply(ctx, [mptr[0]], [sentinel(n, "bf16")], 1.0)
            assert e.value.status == fa.FA_ERR_ARG
        finally:
            torch.cuda.synchronize()
            fa.fa_close(ctx)
    finally:
        torch.cuda.synchronize()
        for f in frees:
            f()


def _free_mib():
    torch.cuda.synchronize()
    free, _ = torch.cuda.mem_get_info()
    return free / 2 ** 20


def test_many_rounds_do_not_grow_memory():
    """200 rounds through one context, mixing device, pinned, pageable and staged-pinned chunks,
    batches and multi-chunk calls, with device and host outputs: device memory does not grow
    after the first rounds (staging is allocated once), and every round is right."""
    rng = np.random.default_rng(71)
    numels = [4096 + 5, 300, 70000]
    K = 3
    xs = [[_f32(rng, n) for n in numels] for _ in range(K)]
    w = [2.0, 3.0, 5.0]
    want = [oracle.fedavg_key(w, [True] * K, [xs[k][p] for k in range(K)], "f32", "f32")[0]
            for p in range(len(numels))]
    dev = [[to_dev(x) for x in row] for row in xs]
    pin = [[to_pinned(x) for x in row] for row in xs]
    ctx = fa.fa_open([(f"k{i}", n) for i, n in enumerate(numels)], "f32", "f32", K,
                     ring_slots=2, slot_bytes=1 << 16)
    outs_dev = [torch.empty(n, dtype=torch.float32, device="cuda") for n in numels]
    outs_host = [np.empty(n, np.float32) for n in numels]
    try:
        def one_round(r):
            fa.fa_reset(ctx)
            mode = r % 4
            for p, n in enumerate(numels):
                if mode == 0:
                    fa.fa_accumulate_batch(ctx, list(range(K)), w, p, 0, [dev[k][p] for k in range(K)], n)
                else:
                    for k in range(K):
                        src = (dev, pin, None)[mode - 1] if mode < 3 else None
                        x = src[k][p] if src is not None else xs[k][p]
                        fa.fa_accumulate(ctx, k, w[k], p, 0, x, n)
            outs = outs_host if r % 2 else outs_dev
            fa.fa_finalize(ctx, outs)
            fa.fa_sync(ctx)
            for p in range(len(numels)):
                got = outs[p] if r % 2 else outs[p].cpu().numpy()
                check_f32(got, want[p], 0.3, K, f"round {r} key {p}")
        for r in range(8):
            one_round(r)
        before = _free_mib()
        for r in range(8, 200):
            one_round(r)
        after = _free_mib()
        assert abs(before - after) < 4, (before, after)
    finally:
        fa.fa_close(ctx)


def test_open_close_cycles_release_everything():
    """Contexts that allocated their sum, staging ring, pinned slots and output staging are
    freed completely by fa_close: 40 open/use/close cycles leave device memory as it was."""
    n = 1 << 20
    x = np.ones(n, np.float32)
    out_host = np.empty(n, np.float32)
    torch.cuda.synchronize()

    def cycle():
        ctx = fa.fa_open([("k", n)], "f32", "f32", 2, ring_slots=2, slot_bytes=1 << 20,
                         flags=fa.FA_STAGE_HOST)
        try:
            fa.fa_accumulate(ctx, 0, 1.0, 0, 0, x, n)                 # pageable: ring + pinned slots
            fa.fa_accumulate(ctx, 1, 1.0, 0, 0, to_pinned(x), n)      # staged pinned
            fa.fa_finalize(ctx, [out_host])                           # host output: output staging
            fa.fa_sync(ctx)
        finally:
            fa.fa_close(ctx)
        assert np.all(out_host == 1.0)

    cycle()
    before = _free_mib()
    for _ in range(40):
        cycle()
    after = _free_mib()
    assert abs(before - after) < 4, (before, after)
