"""Throughput of server-side FedAvg aggregation on GB300.

One step = one aggregation round of the whole path: reset, every client's
update streamed in flat chunks through fa_accumulate (weighted fp32 running
sum in HBM), fa_finalize (divide by the per-key weight total, RNE to bf16).

  value  client-update GB/s with every client's update already resident in HBM
         (the chunks a NIC or copy engine would have landed there)
  e2e    the same metric through the same C ABI calls with pinned HOST buffers:
         every step the kernels read the client updates from host memory in place
         over NVLink-C2C (--stage-host: through the library's staging ring instead)
         and write the aggregate into a pinned host buffer
  roofline  the accumulate kernel (the dominant one): algorithmic bytes per launch
         (bf16 input read + fp32 sum read + fp32 sum write; the first client's
         launches skip the sum read) over its CUDA-event-timed duration
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample
  resident  the same round when every update is resident, reduced in one pass by
         fa_reduce_resident (K*s_in + s_out bytes per element), for comparison: device
         time per round (the host's work hidden behind a queued device-side wait) and wall
         time per round back to back
  compensated  the streamed round in the compensated mode (FA_COMPENSATED: a (hi, lo)
         pair sum, within one bf16 ulp of the exact mean everywhere), its HBM fraction
         on that mode's bytes (s_in + 16 per later client-element)

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica (the path has no exchange
step): value = all ranks' client bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "client-update GB/s aggregated (1×GB300) and % of HBM peak; oracle host GB/s"
# rounds of at most this many client bytes are also timed captured into a CUDA graph and
# replayed (the small, launch-bound models; a 7B round is bound by HBM, not by its calls)
GRAPH_MAX_BYTES = 4 << 30
DEFAULT_WORKLOAD = "llama7b"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------------------- round drivers
def stream_client(fa, ctx, w, k, base_ptr, stream, outs=None):
    """Client k's whole update (flat layout at base_ptr, device or host) in chunk_elems
    pieces; through fa_accumulate_final into `outs` (an fa.out_array) when given."""
    P, ce = w.P, w.chunk_elems or w.P
    es = 2 if w.dtype_in == "bf16" else 4
    calls = 0
    for c0 in range(0, P, ce):
        n = min(ce, P - c0)
        if outs is not None:
            fa.fa_accumulate_final(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0, base_ptr + c0 * es, n, outs,
                                   stream)
        else:
            fa.fa_accumulate(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0, base_ptr + c0 * es, n, stream)
        calls += 1
    return calls


def run_streamed_round(w, resident=False, flags=0, fused=False):
    """One full round on the device, inputs from the device generator, streamed
    client by client exactly as the bench does; returns the flat bf16 output.
    `flags` adds fa_opts flags (FA_COMPENSATED for the compensated mode); `fused` sends the
    last client through fa_accumulate_final, as the bench's timed round does."""
    import torch

    import server_side_fedavg_gb300 as fa
    import synth

    tdt = torch.int16 if w.dtype_in == "bf16" else torch.float32
    s = torch.cuda.current_stream()
    ctx = fa.fa_open([(n, m) for (n, _), m in zip(w.keys, w.numels)], w.dtype_in, w.dtype_out,
                     w.K, flags=fa.FA_FLAT_OUT | flags)
    try:
        if resident:
            bufs = [torch.empty(w.P, dtype=tdt, device="cuda") for _ in range(w.K)]
            for k in range(w.K):
                synth.client_fill_device(w, k, 0, w.P, bufs[k].data_ptr(), s.cuda_stream)
        else:
            buf = torch.empty(w.P, dtype=tdt, device="cuda")
        out = torch.empty(w.P, dtype=torch.int16 if w.dtype_out == "bf16" else torch.float32,
                          device="cuda")
        outs = fa.out_array([out])
        for k in range(w.K):
            if resident:
                ptr = bufs[k].data_ptr()
            else:
                synth.client_fill_device(w, k, 0, w.P, buf.data_ptr(), s.cuda_stream)
                ptr = buf.data_ptr()
            stream_client(fa, ctx, w, k, ptr, s.cuda_stream, outs if fused and k == w.K - 1 else None)
        fa.fa_finalize(ctx, [out], s.cuda_stream)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
        return out
    finally:
        fa.fa_close(ctx)


def run_resident_round(w, flags=0):
    """Every client's full update generated into HBM, then one fa_reduce_resident round
    exactly as the bench's `resident` measurement runs it; returns the flat output."""
    import torch

    import server_side_fedavg_gb300 as fa
    import synth

    tdt = torch.int16 if w.dtype_in == "bf16" else torch.float32
    s = torch.cuda.current_stream()
    bufs = [torch.empty(w.P, dtype=tdt, device="cuda") for _ in range(w.K)]
    for k in range(w.K):
        synth.client_fill_device(w, k, 0, w.P, bufs[k].data_ptr(), s.cuda_stream)
    out = torch.empty(w.P, dtype=torch.int16 if w.dtype_out == "bf16" else torch.float32,
                      device="cuda")
    ctx = fa.fa_open([(n, m) for (n, _), m in zip(w.keys, w.numels)], w.dtype_in, w.dtype_out,
                     w.K, flags=fa.FA_FLAT_OUT | flags)
    try:
        fa.fa_reduce_resident(ctx, list(range(w.K)), w.weights, [b.data_ptr() for b in bufs],
                              [out], s.cuda_stream)
        fa.fa_sync(ctx)
        torch.cuda.synchronize()
    finally:
        fa.fa_close(ctx)
    del bufs
    torch.cuda.empty_cache()
    return out


def partial(w):
    """True when some client sends only part of the keys (an adapter round)."""
    return any(len(r) < w.n_keys for r in w.reports)


def reporters(w):
    """Per key, the number of clients that send it (and its total weight)."""
    cnt = [0] * w.n_keys
    tot = [0.0] * w.n_keys
    for k in range(w.K):
        for p in w.reports[k]:
            cnt[p] += 1
            tot[p] += w.weights[k]
    return cnt, tot


def algorithmic_bytes(w):
    """Per round, streaming path: a key's first reporter s_in+4, later reporters s_in+8,
    finalize 4+s_out bytes per element of every key written (N_p > 0)."""
    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    cnt, tot = reporters(w)
    acc_first = sum(n * (si + 4) for n, c in zip(w.numels, cnt) if c > 0)
    acc_later = sum(n * (c - 1) * (si + 8) for n, c in zip(w.numels, cnt) if c > 1)
    fin = sum(n * (4 + so) for n, t in zip(w.numels, tot) if t > 0)
    return acc_first, acc_later, fin


def resident_kernel(w):
    """The kernel fa_reduce_resident runs for this workload: a layout of more than 48 keys
    from at most 16 clients whose per-key tables fit a launch's 32,640 bytes of table
    parameters (32 B per key, 8 B per client and key, 12 B per client) takes the one-launch
    subset-reduce kernel; otherwise the J-client reduce kernel in final mode."""
    si = "bf16" if w.dtype_in == "bf16" else "f32"
    so = "bf16" if w.dtype_out == "bf16" else "f32"
    nk, K = w.n_keys, w.K
    if K <= 16 and nk > 48 and 32 * nk + 8 * nk * K + 12 * K <= 32640 and max(w.numels) < 2 ** 32:
        return f"reduce_gather_inline_kernel<{si},{so}>"
    return f"reduce_bulk_kernel<{si},{so},final>"


def fused_bytes(w):
    """Per round, streaming path with the last client's chunks through fa_accumulate_final
    (every client sends every key): the first client s_in + 4, the middle ones s_in + 8,
    the last s_in + 4 + s_out (read x and the sum, write the output; no finalize) bytes per
    element."""
    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    return w.P * (si + 4), w.P * (w.K - 2) * (si + 8), w.P * (si + 4 + so)


def subsets_kernel(w):
    """The kernel fa_reduce_subsets runs for this round: the form with its tables in the
    launch's parameters when they fit 32,640 bytes (32 B per key written, 8 B per
    (client, key) entry, 12 B per client), else the one with tables in device memory."""
    si = "bf16" if w.dtype_in == "bf16" else "f32"
    so = "bf16" if w.dtype_out == "bf16" else "f32"
    cnt, tot = reporters(w)
    nseg = sum(1 for c, t in zip(cnt, tot) if c > 0 and t > 0)
    nsrc = sum(len(r) for r in w.reports)
    if 32 * nseg + 8 * nsrc + 12 * w.K <= 32640 and max(w.numels) < 2 ** 32:
        return f"reduce_gather_inline_kernel<{si},{so}>"
    return f"reduce_gather_kernel<{si},{so}>"


def subset_bytes(w):
    """Per round, the one-pass subset reduce: J_p * s_in + s_out per element of every key
    written."""
    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    cnt, tot = reporters(w)
    return sum(n * (c * si + so) for n, c, t in zip(w.numels, cnt, tot) if t > 0)


def packed_offsets(w, k):
    """Element offset of each of client k's keys in its packed buffer (keys back to back
    in report order)."""
    out, o = [], 0
    for p in w.reports[k]:
        out.append(o)
        o += w.numels[p]
    return out, o


def fill_packed(w, k, ptr, stream, es):
    """Client k's reported keys, back to back, generated on the device at ptr."""
    import synth
    offs, _ = packed_offsets(w, k)
    flat = w.flat_offsets()
    for p, o in zip(w.reports[k], offs):
        synth.client_fill_device(w, k, flat[p], w.numels[p], ptr + o * es, stream)


# The source files each kernel family is compiled from: an ncu summary records the digest
# of its kernel's files, so a figure taken on an older kernel is never reported as current.
KERNEL_SOURCES = {
    "accumulate": ("kernels.cuh", "device.cuh", "tiles.hpp", "accumulate.cu"),
    "reduce": ("kernels.cuh", "device.cuh", "tiles.hpp", "reduce.cu"),
    "gather": ("kernels.cuh", "gather.cuh", "device.cuh", "tiles.hpp", "gather.cu", "gather_plan.cpp"),
    "finalize": ("kernels.cuh", "device.cuh", "tiles.hpp", "finalize.cu"),
}


def kernel_source_digest(sources=None):
    """sha256 (first 16 hex digits) of the named kernel sources (default: every family's)."""
    import hashlib
    if sources is None:
        sources = sorted({f for fs in KERNEL_SOURCES.values() for f in fs})
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "server_side_fedavg_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(bytes_per_launch):
    """DRAM bytes per accumulate launch from the committed ncu figures
    (profiles/accumulate_decoder1l.json), scaled from the captured launch to the average
    launch by algorithmic bytes; None once the kernel's sources differ from the ones the
    counters were taken on."""
    path = os.path.join(ROOT, "profiles", "accumulate_decoder1l.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_digest") != kernel_source_digest(d["sources"]):
            return None
        dram = float(d["dram_bytes_per_launch"])
        algo = float(d["algorithmic_bytes_of_captured_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None
    return int(dram / algo * bytes_per_launch)


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        # nvidia-smi addresses the GPU by UUID: its indexes need not match CUDA's when
        # CUDA_VISIBLE_DEVICES remaps them
        self.gpu = str(device)
        try:
            import torch
            uuid = getattr(torch.cuda.get_device_properties(device), "uuid", None)
            if uuid is not None:
                self.gpu = f"GPU-{uuid}"
        except Exception:  # pragma: no cover - property missing in this torch
            pass
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="fedavg_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- CPU oracle baseline
def cpu_sample(w, elems):
    """Inputs of the CPU sample: the first `elems` flat elements of every client."""
    import synth
    return [synth.client_flat(w, k, 0, elems) for k in range(w.K)]


def cpu_pass(w, xs, threads):
    """One timed pass of the fp64 oracle (as it stands) over the sample, split
    into contiguous slices over `threads` host threads (ctypes drops the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    elems = xs[0].size
    per = -(-elems // threads)
    reps = [True] * w.K

    def part(i):
        a, b = i * per, min(elems, (i + 1) * per)
        if b > a:
            oracle.fedavg_key(w.weights, reps, [x[a:b] for x in xs], w.dtype_in, w.dtype_out)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(part, range(threads)))
    return time.perf_counter() - t0


def cpu_baseline(w, elems, min_seconds=10.0, threads=None, min_seconds_1t=3.0):
    """Oracle throughput on the host cores: passes over a bounded sample until
    at least `min_seconds` of wall time; inputs are made before timing.  The same
    oracle on one thread (a quarter of the sample, at least `min_seconds_1t`) is
    reported beside it."""
    threads = threads or (os.cpu_count() or 1)
    xs = cpu_sample(w, elems)
    si = 2 if w.dtype_in == "bf16" else 4
    passes, dt = 0, 0.0
    while dt < min_seconds:
        dt += cpu_pass(w, xs, threads)
        passes += 1
    gbs = passes * w.K * elems * si / dt / 1e9
    q = max(1, elems // 4)
    xq = [x[:q] for x in xs]
    p1, dt1 = 0, 0.0
    while dt1 < min_seconds_1t:
        dt1 += cpu_pass(w, xq, 1)
        p1 += 1
    gbs1 = p1 * w.K * q * si / dt1 / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "value_1thread": round(gbs1, 3),
            "sample": f"{w.name}: first {elems} flat elements x {w.K} clients "
                      f"({w.K * elems * si / 1e9:.2f} GB of client bytes), fp64 C oracle, "
                      f"{passes} passes in {dt:.1f} s on {threads} threads; 1 thread: first {q} "
                      f"elements, {p1} passes in {dt1:.1f} s"}


def partition_plan_us(m, reps=20000):
    """Host time of one fa_partition_plan call for m participants (the library call itself:
    arrays are built once), in microseconds."""
    import ctypes

    import server_side_fedavg_gb300 as fa
    rng = np.random.default_rng(0)
    t = rng.uniform(1.0, 2.0, m)
    e = rng.uniform(1.0, 2.0, m)
    n = rng.integers(100, 1000, m).astype(np.uint64)
    tau = np.full(m, np.nan)
    eps = np.full(m, np.nan)
    out = np.zeros(m, np.uint64)
    opts = fa.fa_partition_opts(1.0, 0.0, 0.5, 0.05)
    lib = fa.lib()
    args = (m, t.ctypes.data, e.ctypes.data, n.ctypes.data, tau.ctypes.data, eps.ctypes.data,
            ctypes.byref(opts), out.ctypes.data)
    assert lib.fa_partition_plan(*args) == 0
    t0 = time.perf_counter()
    for _ in range(reps):
        lib.fa_partition_plan(*args)
    return round((time.perf_counter() - t0) / reps * 1e6, 3)


# --------------------------------------------------------------------------- distributed bits
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        if torch.cuda.is_available():
            torch.cuda.set_device(local)          # one GPU per rank, bound before NCCL starts
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        import torch
        if pg.get_backend() == "nccl":
            pg.barrier(device_ids=[torch.cuda.current_device()])
        else:
            pg.barrier()


def max_over_ranks(pg, v: float) -> float:
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- arms
def run_reference(args, world, rank, pg):
    from synth import workloads as W

    if rank != 0:
        return 0
    w = W.make(args.workload)
    elems = args.ref_elems
    threads = os.cpu_count() or 1
    si = 2 if w.dtype_in == "bf16" else 4
    xs = cpu_sample(w, elems)
    for _ in range(args.warmup):
        cpu_pass(w, xs, threads)
    times = [cpu_pass(w, xs, threads) for _ in range(args.steps)]
    v = round(w.K * elems * si * args.steps / sum(times) / 1e9, 3)
    sample = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
              "sample": f"{w.name}: first {elems} flat elements x {w.K} clients "
                        f"({w.K * elems * si / 1e9:.2f} GB of client bytes) per step, "
                        f"fp64 C oracle on {threads} threads"}
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sum(times) / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "K": w.K, "P": w.P, "sample_elems": elems},
        "cpu_baseline": sample,
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local, pg):
    import torch

    import server_side_fedavg_gb300 as fa
    import synth
    from synth import workloads as W

    torch.cuda.set_device(local)
    w = W.make(args.workload)
    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    tin = torch.int16 if si == 2 else torch.float32
    tout = torch.int16 if so == 2 else torch.float32
    layout = [(n, m) for (n, _), m in zip(w.keys, w.numels)]
    s = torch.cuda.Stream()
    sh = s.cuda_stream
    client_bytes = w.client_bytes()
    peak, peak_kind = _peaks()
    part = partial(w)

    # ---- regime A: every client's update resident in HBM (for an adapter round, each
    # client's reported keys packed back to back)
    free, _ = torch.cuda.mem_get_info()
    per_client = w.P * si
    fixed = w.P * 4 + w.P * so + (6 << 30)
    resident = w.K if part else max(1, min(w.K, int((free - fixed) // per_client)))
    if part:
        bufs = [torch.empty(max(1, packed_offsets(w, k)[1]), dtype=tin, device="cuda") for k in range(w.K)]
        for k in range(w.K):
            fill_packed(w, k, bufs[k].data_ptr(), sh, si)
        import numpy as _np
        key_args = []
        for k in range(w.K):
            offs, _ = packed_offsets(w, k)
            key_args.append((_np.asarray(w.reports[k], _np.int64), _np.zeros(len(offs), _np.uint64),
                             _np.asarray([bufs[k].data_ptr() + o * si for o in offs], _np.uint64),
                             _np.asarray([w.numels[p] for p in w.reports[k]], _np.uint64)))
    else:
        bufs = [torch.empty(w.P, dtype=tin, device="cuda") for _ in range(resident)]
        for k in range(resident):
            synth.client_fill_device(w, k, 0, w.P, bufs[k].data_ptr(), sh)
    out = torch.empty(w.P, dtype=tout, device="cuda")
    ctx = fa.fa_open(layout, w.dtype_in, w.dtype_out, w.K, flags=fa.FA_FLAT_OUT)
    torch.cuda.synchronize()

    nchunk = -(-w.P // (w.chunk_elems or w.P))

    # the last client's chunks go through fa_accumulate_final (its kernels write the
    # aggregate; fa_finalize then has nothing left to write) unless --no-fused, or when
    # clients send key subsets (then fa_accumulate_keys and fa_finalize)
    fused = not part and not args.no_fused and w.K >= 2
    out_arr = fa.out_array([out])

    def step(evs=None, final=fused, sh=sh, reset=True):
        # evs: (start, after the accumulate launches, after finalize, after clients 0..K-2)
        # on the launching stream
        if reset:
            fa.fa_reset(ctx)
        if evs is not None:
            evs[0].record(s)
        for k in range(w.K):
            if evs is not None and k == w.K - 1:
                evs[3].record(s)
            if part:
                ks, os_, ps, ls = key_args[k]
                fa.fa_accumulate_keys(ctx, k, w.weights[k], ks, os_, ps, ls, sh)
                continue
            base = bufs[k % resident].data_ptr()
            P, ce = w.P, w.chunk_elems or w.P
            last = final and k == w.K - 1
            for c0 in range(0, P, ce):
                if last:
                    fa.fa_accumulate_final(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0, base + c0 * si,
                                           min(ce, P - c0), out_arr, sh)
                else:
                    fa.fa_accumulate(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0, base + c0 * si,
                                     min(ce, P - c0), sh)
        if evs is not None:
            evs[1].record(s)
        fa.fa_finalize(ctx, [out], sh)
        if evs is not None:
            evs[2].record(s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()

    n_calls = w.K * nchunk          # accumulate launches per round (flat chunks)
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = fa.fa_get_stats(ctx)["kernel_launches"]
    clocks = ClockSampler(local)
    clocks.start()
    t0e.record(s)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        step(ev_sets[i])
    t1e.record(s)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    launches = fa.fa_get_stats(ctx)["kernel_launches"] - launches0
    if part:
        n_calls = max(1, launches // args.steps - 1)   # accumulate launches (all but finalize)
    barrier(pg)
    ms_total = t0e.elapsed_time(t1e)
    ms_total = max_over_ranks(pg, ms_total)

    # kernel times: events bracket each step's run of accumulate launches (one launch
    # per call here) and its finalize launch, on the stream they are launched on
    acc_ms = 0.0
    fin_ms = 0.0
    last_ms = 0.0          # the last client's launches (the final form in a fused round)
    for evs in ev_sets:
        acc_ms += evs[0].elapsed_time(evs[1])
        fin_ms += evs[1].elapsed_time(evs[2])
        last_ms += evs[3].elapsed_time(evs[1])
    final_form = None
    if fused:
        b0, b1, b2 = fused_bytes(w)
        step_bytes = b0 + b1 + b2
        # the dominant launches are the plain form's (clients 0..K-2); the last client's
        # final-form launches are reported beside them
        acc_bytes = b0 + b1
        acc_ms -= last_ms
        n_calls = (w.K - 1) * nchunk
        fl = nchunk
        f_launch_ms = last_ms / (args.steps * fl)
        f_ach = b2 / fl / (f_launch_ms * 1e-3) / 1e9
        final_form = {"kernel": f"accumulate_bulk_kernel<{w.dtype_in}, final, {w.dtype_out}>",
                      "achieved": round(f_ach, 1), "frac": round(f_ach / peak, 4),
                      "bytes_per_launch": int(b2 / fl), "launch_ms": round(f_launch_ms, 4)}
    else:
        acc_first_b, acc_later_b, fin_b = algorithmic_bytes(w)
        acc_bytes = acc_first_b + acc_later_b
        step_bytes = acc_bytes + fin_b
    acc_launch_ms = acc_ms / (args.steps * n_calls)
    acc_bytes_per_launch = acc_bytes / n_calls
    achieved = acc_bytes_per_launch / (acc_launch_ms * 1e-3) / 1e9
    ms_per_step = ms_total / args.steps
    value = world * client_bytes / (ms_per_step * 1e-3) / 1e9

    # ---- the same round with every client through fa_accumulate and then fa_finalize:
    # the finalize kernel's rate, and the sum a delta round's finalize reads below
    unfused_line = None
    ev_u = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for _ in range(2 if fused else 0):
        step(final=False)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if fused:
        u0.record(s)
        for i in range(args.steps):
            step(ev_u[i], final=False)
        u1.record(s)
        torch.cuda.synchronize()
        ums = max_over_ranks(pg, u0.elapsed_time(u1)) / args.steps
        ufin = sum(e[1].elapsed_time(e[2]) for e in ev_u) / args.steps
        _, _, fin_b = algorithmic_bytes(w)
        fin_gbs = fin_b / (ufin * 1e-3) / 1e9
        unfused_line = {"value": round(world * client_bytes / (ums * 1e-3) / 1e9, 2), "unit": "GB/s",
                        "ms_per_step": round(ums, 3), "finalize_ms": round(ufin, 3),
                        "calls": "every client through fa_accumulate, then fa_finalize"}
    else:
        fin_gbs = fin_b / (fin_ms / args.steps * 1e-3) / 1e9

    # ---- a launch-bound round (a small model) captured once into a CUDA graph and replayed:
    # the host's calls leave the round, one graph launch remains
    graph_line = None
    if not args.no_graph and client_bytes <= GRAPH_MAX_BYTES:
        graph_line = graph_replay(fa, ctx, lambda gsh: step(sh=gsh, reset=False), max(20, args.steps))
        graph_line["calls_wall_ms_per_round"] = round(wall / args.steps * 1e3, 4)
        graph_line["value"] = round(world * client_bytes / (graph_line["wall_ms_per_round"] * 1e-3) / 1e9, 2)
        graph_line["unit"] = "GB/s"
        step(final=False)   # the delta-round finalize below reads this round's sum

    # ---- a delta round's finalize: the same aggregate applied in place to a base model
    # (fa_finalize_apply, server_lr 0.5): reads the sum and the base, writes the output
    for _ in range(2):
        fa.fa_finalize_apply(ctx, [out], [out], 0.5, sh)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(s)
    for _ in range(args.steps):
        fa.fa_finalize_apply(ctx, [out], [out], 0.5, sh)
    a1.record(s)
    torch.cuda.synchronize()
    ams = a0.elapsed_time(a1) / args.steps
    abytes = w.P * (4 + 2 * so)
    apply_line = {"gbs": round(abytes / (ams * 1e-3) / 1e9, 1),
                  "frac": round(abytes / (ams * 1e-3) / 1e9 / peak, 4), "ms": round(ams, 3),
                  "bytes": int(abytes), "kernel": f"finalize_kernel<{w.dtype_out},apply>"}

    # ---- the same round with every update resident, reduced in one pass (fa_reduce_resident)
    resident_line = None
    subsets_line = None
    if part and not args.no_resident:
        subsets_line = run_subsets(args, w, ctx, bufs, out, s, peak)
    if resident == w.K and not part and not args.no_resident:
        ids = list(range(w.K))
        ptrs = [b.data_ptr() for b in bufs]

        def round_resident(e=None):
            fa.fa_reset(ctx)
            if e is not None:
                # a short device-side wait ahead of the call, so that the call's host work is
                # done before the GPU reaches the start event: the events bracket device work
                with torch.cuda.stream(s):
                    torch.cuda._sleep(4_000_000)
                e[0].record(s)
            fa.fa_reduce_resident(ctx, ids, w.weights, ptrs, [out], sh)
            if e is not None:
                e[1].record(s)

        for _ in range(args.warmup):
            round_resident()
        torch.cuda.synchronize()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0 = fa.fa_get_stats(ctx)["kernel_launches"]
        r0.record(s)
        for _ in range(args.steps):
            round_resident()
        r1.record(s)
        torch.cuda.synchronize()
        wall_ms = r0.elapsed_time(r1) / args.steps
        launches_r = int((fa.fa_get_stats(ctx)["kernel_launches"] - l0) // args.steps)
        evr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for e in evr:
            round_resident(e)
        torch.cuda.synchronize()
        rms = sum(a.elapsed_time(b) for a, b in evr) / len(evr)
        rbytes = w.P * (w.K * si + so)
        rgraph = None
        if not args.no_graph and client_bytes <= GRAPH_MAX_BYTES:
            rgraph = graph_replay(fa, ctx, lambda sh: fa.fa_reduce_resident(ctx, ids, w.weights, ptrs, [out], sh),
                                  max(20, args.steps))
            rgraph["hbm_frac"] = round(rbytes / (rgraph["device_ms_per_round"] * 1e-3) / 1e9 / peak, 4)
        resident_line = {"value": round(client_bytes / (rms * 1e-3) / 1e9, 2), "unit": "GB/s",
                         "device_ms_per_round": round(rms, 4), "wall_ms_per_round": round(wall_ms, 4),
                         "value_wall": round(client_bytes / (wall_ms * 1e-3) / 1e9, 2),
                         "hbm_gbs": round(rbytes / (rms * 1e-3) / 1e9, 1),
                         "hbm_frac": round(rbytes / (rms * 1e-3) / 1e9 / peak, 4),
                         "bytes_per_round": int(rbytes), "launches_per_round": launches_r,
                         "graph": rgraph,
                         "kernel": resident_kernel(w)}

    fa.fa_close(ctx)
    torch.cuda.synchronize()

    # ---- the same streamed round in the compensated mode (FA_COMPENSATED): the running sum
    # is a (hi, lo) pair, so each later client-element moves 8 more bytes
    comp_line = None
    if not args.no_compensated and not part:
        comp_line = run_compensated(args, w, layout, bufs, out, s, peak)

    del bufs, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # ---- e2e: pinned host buffers through the same calls
    e2e = None
    if args.e2e_steps > 0:
        hb = e2e_buffers(args, w, world)
        e2e = run_e2e(args, w, layout, s, pg, world, hb)
        if args.e2e_staged_steps > 0 and not args.stage_host:
            # the same end-to-end round through the library's staging ring (FA_STAGE_HOST:
            # copies on a copy stream into device slots, then the accumulate kernel)
            import argparse
            a2 = argparse.Namespace(**vars(args))
            a2.stage_host = True
            a2.e2e_steps = args.e2e_staged_steps
            st = run_e2e(a2, w, layout, s, pg, world, hb)
            e2e["staged"] = {k: st[k] for k in ("value", "ms_per_step", "accumulate_ms", "finalize_ms",
                                                 "host_call_ms", "host_cpu_ms", "link_frac",
                                                 "accumulate_link_frac", "ingest", "output")}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "P": w.P, "K": w.K, "n_keys": w.n_keys,
                   "dtype_in": w.dtype_in, "dtype_out": w.dtype_out,
                   "chunk_bytes": (w.chunk_elems or w.P) * si, "resident_clients": resident,
                   "l2": "inputs (client updates, running sum) far larger than L2; no flush",
                   "hbm_frac_step": round(step_bytes / (ms_per_step * 1e-3) / 1e9 / peak, 4),
                   "finalize_gbs": round(fin_gbs, 1),
                   "last_client": ("fa_accumulate_final (its kernels write the aggregate)" if fused
                                   else "fa_accumulate, then fa_finalize"),
                   "wall_s": round(wall, 3)},
        "roofline": {"bound": "hbm",
                     "kernel": (f"accumulate_bulk_kernel<{w.dtype_in}> (clients 0..{w.K - 2}; the last "
                                f"client's final form in final_form)" if fused
                                else f"accumulate_bulk_kernel<{w.dtype_in}>"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "bytes_per_launch": int(acc_bytes_per_launch),
                     "launch_ms": round(acc_launch_ms, 4),
                     "traffic": profiled_traffic(acc_bytes_per_launch),
                     "final_form": final_form},
        "gpu_launches": int(launches),
        "unfused": unfused_line,
        "graph": graph_line,
        "resident": resident_line,
        "subsets": subsets_line,
        "compensated": comp_line,
        "delta_apply": apply_line,
        "partition_plan_us": partition_plan_us(w.K),
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.ref_elems)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def graph_replay(fa, ctx, calls, reps):
    """A round captured once into a CUDA graph and replayed `reps` times back to back on
    the current stream: wall and device (CUDA events) ms per replayed round.  calls(stream)
    issues the round's library calls on the capturing stream; fa_reset runs before the
    capture (it waits for the context's work) and after it, leaving the context as it was."""
    import torch

    fa.fa_reset(ctx)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    cs = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    t0 = time.perf_counter()
    for _ in range(reps):
        g.replay()
    e1.record(cs)
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) / reps
    dev = e0.elapsed_time(e1) / reps
    del g
    fa.fa_reset(ctx)
    return {"wall_ms_per_round": round(wall * 1e3, 4), "device_ms_per_round": round(dev, 4)}


def run_subsets(args, w, ctx, bufs, out, s, peak):
    """An adapter round through fa_reduce_subsets (each client's reported keys, packed in
    its resident buffer, reduced straight to the output): device time on the stream (CUDA
    events around the call's table upload and kernel, with the host's work hidden behind
    a device-side wait queued first) and wall time per round, back to back (the host
    bookkeeping of every (client, key) entry and fa_reset's wait included)."""
    import torch

    import server_side_fedavg_gb300 as fa

    ids = list(range(w.K))
    ptrs = [b.data_ptr() for b in bufs]
    table = fa.subset_table(w.reports)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(max(1, args.steps))]

    def round_(e=None):
        fa.fa_reset(ctx)
        if e is not None:
            # a short device-side wait ahead of the call, so that the call's host work is done
            # before the GPU reaches the start event: the events then bracket device work only
            with torch.cuda.stream(s):
                torch.cuda._sleep(4_000_000)
            e[0].record(s)
        fa.fa_reduce_subsets(ctx, ids, w.weights, ptrs, table, [out], s.cuda_stream)
        if e is not None:
            e[1].record(s)

    for _ in range(max(3, args.warmup)):
        round_()
    torch.cuda.synchronize()
    l0 = fa.fa_get_stats(ctx)["kernel_launches"]
    t0 = time.perf_counter()
    for _ in range(len(ev)):
        round_()
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) / len(ev)
    launches = (fa.fa_get_stats(ctx)["kernel_launches"] - l0) // len(ev)
    for e in ev:
        round_(e)
    torch.cuda.synchronize()
    dev_ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    b = subset_bytes(w)
    cb = w.client_bytes()
    graph = None if args.no_graph else graph_replay(
        fa, ctx, lambda sh: fa.fa_reduce_subsets(ctx, ids, w.weights, ptrs, table, [out], sh),
        max(20, args.steps))
    if graph is not None:
        graph["hbm_frac"] = round(b / (graph["device_ms_per_round"] * 1e-3) / 1e9 / peak, 4)
    return {"value": round(cb / (dev_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "device_ms_per_round": round(dev_ms, 4), "wall_ms_per_round": round(wall * 1e3, 4),
            "value_wall": round(cb / wall / 1e9, 2),
            "hbm_gbs": round(b / (dev_ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(b / (dev_ms * 1e-3) / 1e9 / peak, 4),
            "bytes_per_round": int(b), "launches_per_round": int(launches),
            "graph": graph,
            "kernel": subsets_kernel(w)}


def run_compensated(args, w, layout, bufs, out, s, peak):
    """The bench's streamed round with FA_COMPENSATED: client-update GB/s, the round's
    algorithmic HBM bytes (first client s_in + 8, later ones s_in + 16, finalize 8 + s_out
    per element) over its time, and the accumulate launches' own fraction.  The pair sum
    takes twice the default sum's memory: if the resident client buffers leave no room for
    it, the last ones are dropped and clients reuse the remaining buffers (each read is
    still a fresh pass over a buffer far larger than L2)."""
    import torch

    import server_side_fedavg_gb300 as fa

    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    sh = s.cuda_stream
    pad = sum(-(-n // 32) * 32 for n in w.numels)
    need = 2 * pad * 4 + (4 << 30)
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    bufs = list(bufs)
    while free < need and len(bufs) > 1:
        bufs.pop()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        free, _ = torch.cuda.mem_get_info()
    if free < need:
        return {"skipped": "no device memory for the pair sum"}
    ctx = fa.fa_open(layout, w.dtype_in, w.dtype_out, w.K, flags=fa.FA_FLAT_OUT | fa.FA_COMPENSATED)
    try:
        ce = w.chunk_elems or w.P
        nchunk = -(-w.P // ce)

        def step(evs=None):
            fa.fa_reset(ctx)
            if evs is not None:
                evs[0].record(s)
            for k in range(w.K):
                base = bufs[k % len(bufs)].data_ptr()
                for c0 in range(0, w.P, ce):
                    fa.fa_accumulate(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0, base + c0 * si,
                                     min(ce, w.P - c0), sh)
            if evs is not None:
                evs[1].record(s)
            fa.fa_finalize(ctx, [out], sh)
            if evs is not None:
                evs[2].record(s)

        for _ in range(max(1, args.warmup)):
            step()
        torch.cuda.synchronize()
        steps = max(1, args.steps)
        ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            step(ev_sets[i])
        torch.cuda.synchronize()
        acc_ms = sum(e[0].elapsed_time(e[1]) for e in ev_sets) / steps
        fin_ms = sum(e[1].elapsed_time(e[2]) for e in ev_sets) / steps
        round_ms = sum(e[0].elapsed_time(e[2]) for e in ev_sets) / steps
    finally:
        fa.fa_close(ctx)
    acc_b = w.P * (si + 8) + (w.K - 1) * w.P * (si + 16)
    fin_b = w.P * (8 + so)
    acc_gbs = acc_b / (acc_ms * 1e-3) / 1e9
    return {"value": round(w.K * w.P * si / (round_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_round": round(round_ms, 3),
            "hbm_gbs": round((acc_b + fin_b) / (round_ms * 1e-3) / 1e9, 1),
            "hbm_frac": round((acc_b + fin_b) / (round_ms * 1e-3) / 1e9 / peak, 4),
            "bytes_per_round": int(acc_b + fin_b),
            "accumulate": {"kernel": f"accumulate_bulk_kernel<{w.dtype_in},compensated>",
                           "achieved": round(acc_gbs, 1), "frac": round(acc_gbs / peak, 4),
                           "bytes_per_launch": int(acc_b / (w.K * nchunk)),
                           "launch_ms": round(acc_ms / (w.K * nchunk), 4)},
            "finalize_gbs": round(fin_b / (fin_ms * 1e-3) / 1e9, 1),
            "distinct_client_buffers": len(bufs)}


def host_mem_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def h2d_peak(src, s, reps=8):
    """Plain pinned-host -> device copy rate of one buffer (GB/s, CUDA events on s):
    the host link's ceiling for the end-to-end number."""
    import torch
    dst = torch.empty_like(src, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        dst.copy_(src, non_blocking=True)
        e0.record(s)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        e1.record(s)
    e1.synchronize()
    nbytes = src.numel() * src.element_size()
    return reps * nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9


def e2e_buffers(args, w, world):
    """The host side of the end-to-end rounds: client chunks in pinned host memory (a
    pool of distinct chunks, reused) and the output buffer, allocated once and shared by
    the in-place and the staged variants.  Pinned memory is sized to this rank's share
    of the node's available memory (ranks on one node share it); if it does not fit,
    the pool shrinks and the output falls back to pageable memory."""
    import torch

    import synth

    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    ce = w.chunk_elems or w.P
    nchunk = -(-w.P // ce)
    pool_n = min(args.e2e_pool, w.K * nchunk)
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", str(world)))
    avail = host_mem_available()
    budget = None if avail is None else int(0.4 * avail / max(1, local_world))
    out_pinned = True
    if budget is not None:
        out_bytes = w.P * so
        while pool_n > 2 and pool_n * ce * si + out_bytes > budget:
            pool_n //= 2
        if pool_n * ce * si + out_bytes > budget:
            out_pinned = False
    part = partial(w)
    pool = []
    key_args = None
    if part:
        # an adapter round: each client's reported keys packed in one pinned buffer, sent
        # with one fa_accumulate_keys call (read in place over the link)
        import numpy as _np
        pool_n = w.K
        flat = w.flat_offsets()
        key_args = []
        for k in range(w.K):
            offs, tot = packed_offsets(w, k)
            t = torch.empty(max(1, tot), dtype=torch.int16 if si == 2 else torch.float32).pin_memory()
            tv = t.numpy().view(_np.uint16 if si == 2 else _np.float32)
            for p_, o in zip(w.reports[k], offs):
                synth.client_flat(w, k, flat[p_], w.numels[p_], out=tv[o:o + w.numels[p_]])
            pool.append(t)
            key_args.append((_np.asarray(w.reports[k], _np.int64), _np.zeros(len(offs), _np.uint64),
                             _np.asarray([t.data_ptr() + o * si for o in offs], _np.uint64),
                             _np.asarray([w.numels[p_] for p_ in w.reports[k]], _np.uint64)))
    for i in range(0 if part else pool_n):
        k, c = divmod(i, nchunk)
        c0 = c * ce
        n = min(ce, w.P - c0)
        t = torch.empty(ce, dtype=torch.int16 if si == 2 else torch.float32).pin_memory()
        a = synth.client_flat(w, k, c0, n)
        t[:n].numpy().view(a.dtype)[:] = a
        pool.append(t)
    out = torch.empty(w.P, dtype=torch.int16 if so == 2 else torch.float32)
    if out_pinned:
        out = out.pin_memory()
    return {"pool": pool, "pool_n": pool_n, "out": out, "out_pinned": out_pinned, "part": part,
            "key_args": key_args if part else None}


def run_e2e(args, w, layout, s, pg, world, hb):
    """One end-to-end variant over the buffers of e2e_buffers: every step reads the
    client chunks from host memory and writes the aggregate to the host buffer, copies
    inside the timed region."""
    import torch

    import server_side_fedavg_gb300 as fa

    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    ce = w.chunk_elems or w.P
    pool, pool_n, out, out_pinned, part = hb["pool"], hb["pool_n"], hb["out"], hb["out_pinned"], hb["part"]
    key_args = hb["key_args"]
    flags = fa.FA_FLAT_OUT | (fa.FA_STAGE_HOST if args.stage_host else 0)
    ctx = fa.fa_open(layout, w.dtype_in, w.dtype_out, w.K, flags=flags,
                     ring_slots=args.ring_slots, slot_bytes=args.slot_mb << 20)
    sh = s.cuda_stream
    link = h2d_peak(pool[0], s)
    # the last client through fa_accumulate_final: its kernels read its chunks in place and
    # write the aggregate into the pinned output (not for staged chunks or a pageable output)
    fused = (not part and not args.stage_host and not args.no_fused and out_pinned and w.K >= 2)
    out_arr = fa.out_array([out])

    host = {"wall": 0.0, "cpu": 0.0}   # the calling thread's time in the accumulate calls

    def step(evs=None):
        # evs: (start, after the accumulate calls, after finalize) on the stream
        fa.fa_reset(ctx)
        if evs is not None:
            evs[0].record(s)
        i = 0
        hw0, hc0 = time.perf_counter(), time.thread_time()
        for k in range(w.K):
            if part:
                ks, os_, ps, ls = key_args[k]
                if args.stage_host:     # staged host chunks go through fa_accumulate
                    for p_, ptr, n in zip(ks, ps, ls):
                        fa.fa_accumulate(ctx, k, w.weights[k], int(p_), 0, int(ptr), int(n), sh)
                else:
                    fa.fa_accumulate_keys(ctx, k, w.weights[k], ks, os_, ps, ls, sh)
                continue
            for c0 in range(0, w.P, ce):
                n = min(ce, w.P - c0)
                if fused and k == w.K - 1:
                    fa.fa_accumulate_final(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0,
                                           pool[i % pool_n].data_ptr(), n, out_arr, sh)
                else:
                    fa.fa_accumulate(ctx, k, w.weights[k], fa.FA_KEY_FLAT, c0,
                                     pool[i % pool_n].data_ptr(), n, sh)
                i += 1
        if evs is not None:
            host["wall"] += time.perf_counter() - hw0
            host["cpu"] += time.thread_time() - hc0
            evs[1].record(s)
        fa.fa_finalize(ctx, [out], sh)
        if evs is not None:
            evs[2].record(s)
        fa.fa_sync(ctx)

    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.e2e_steps)]
    try:
        for _ in range(max(1, args.warmup // 2)):
            step()
        torch.cuda.synchronize()
        barrier(pg)
        st0 = fa.fa_get_stats(ctx)
        t0 = time.perf_counter()
        for i in range(args.e2e_steps):
            step(ev_sets[i])
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        st1 = fa.fa_get_stats(ctx)
        dt = max_over_ranks(pg, dt)
    finally:
        fa.fa_close(ctx)
    acc_ms = sum(e[0].elapsed_time(e[1]) for e in ev_sets) / args.e2e_steps
    fin_ms = sum(e[1].elapsed_time(e[2]) for e in ev_sets) / args.e2e_steps
    h2d = (st1["h2d_bytes"] - st0["h2d_bytes"]) // args.e2e_steps
    d2h = (st1["d2h_bytes"] - st0["d2h_bytes"]) // args.e2e_steps
    v = world * w.client_bytes() * args.e2e_steps / dt / 1e9
    # HBM traffic of the host-fed round: the running sum (written by a key's first reporter,
    # read and written by every later one, read by finalize); staging adds each chunk's
    # write and read in HBM, and a staged output its device copy (written, then read by the
    # copy)
    a_first, a_later, a_fin = algorithmic_bytes(w)
    hbm = a_first // (si + 4) * 4 + a_later // (si + 8) * 8 + a_fin // (4 + so) * 4
    if fused:   # the last client reads the sum and writes no sum; no finalize reads it
        hbm = w.P * 4 + w.P * (w.K - 2) * 8 + w.P * 4
    if args.stage_host:
        hbm += w.client_bytes() * 2
    if args.stage_host or not out_pinned:
        hbm += 2 * w.P * so
    peak, _ = _peaks()
    return {"value": round(v, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps,
            "ms_per_step": round(dt / args.e2e_steps * 1e3, 2),
            "accumulate_ms": round(acc_ms, 3), "finalize_ms": round(fin_ms, 3),
            "host_call_ms": round(host["wall"] * 1e3 / args.e2e_steps, 1),
            "host_cpu_ms": round(host["cpu"] * 1e3 / args.e2e_steps, 1),
            "h2d_peak_gbs": round(link, 1),
            "link_frac": round(h2d * args.e2e_steps / dt / 1e9 / link, 3),
            "accumulate_link_frac": round(h2d / (acc_ms * 1e-3) / 1e9 / link, 3),
            "hbm_gbs": round(hbm * args.e2e_steps / dt / 1e9, 1),
            "hbm_frac": round(hbm * args.e2e_steps / dt / 1e9 / peak, 4),
            "host_pool": (f"{w.K} pinned buffers, one per client, its reported keys packed" if part
                          else f"{pool_n} distinct pinned chunks of {ce * si >> 20} MiB, reused"),
            "output": (("pinned host buffer, " + ("copied from a device buffer" if args.stage_host
                                                  else "written in place by the last client's kernels"
                                                  if fused else "written in place by the finalize kernel"))
                       if out_pinned else "pageable host buffer (pinned budget too small)"),
            "ingest": (f"staging ring: {args.ring_slots or 4} device slots of {args.slot_mb or 64} MiB"
                       if args.stage_host else "pinned chunks read in place by the accumulate kernel"),
            "last_client": ("fa_accumulate_final: its kernels write the aggregate into the pinned output"
                            if fused else "fa_accumulate, then fa_finalize")}


def run_hierarchical(args, world, rank, local, pg):
    """Two-level FedAvg (silos, then a FedAvg over the silos' fp32 means weighted by each
    silo's total): S silos of K/S clients each.  One step = one two-level round; value =
    client-update GB/s.  Prints its own JSON line ("mode": "hierarchical")."""
    import torch

    import server_side_fedavg_gb300 as fa
    import synth
    from synth import workloads as W

    torch.cuda.set_device(local)
    w = W.make(args.workload)
    S = args.hierarchical
    if w.K % S:
        raise SystemExit(f"{w.K} clients do not split into {S} silos")
    if w.dtype_in != "bf16":
        raise SystemExit("the hierarchical mode streams bf16 client updates")
    per = w.K // S
    layout = [(name, n) for (name, _), n in zip(w.keys, w.numels)]
    s = torch.cuda.Stream()
    sh = s.cuda_stream
    peak, peak_kind = _peaks()
    need = w.K * w.P * 2 + S * w.P * 4 + 2 * w.P * 4 + w.P * 2 + (6 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        raise SystemExit(f"{w.name} with {S} silos needs {need / 1e9:.0f} GB of HBM, {free / 1e9:.0f} free")
    bufs = [torch.empty(w.P, dtype=torch.int16, device="cuda") for _ in range(w.K)]
    for k in range(w.K):
        synth.client_fill_device(w, k, 0, w.P, bufs[k].data_ptr(), sh)
    means = [torch.empty(w.P, dtype=torch.float32, device="cuda") for _ in range(S)]
    out = torch.empty(w.P, dtype=torch.int16, device="cuda")
    silo = fa.fa_open(layout, "bf16", "f32", per, flags=fa.FA_FLAT_OUT)
    top = fa.fa_open(layout, "f32", "bf16", S, flags=fa.FA_FLAT_OUT)
    ce = w.chunk_elems or w.P
    totals = [sum(w.weights[g * per:(g + 1) * per]) for g in range(S)]

    def step():
        for g in range(S):
            fa.fa_reset(silo)
            for j in range(per):
                k = g * per + j
                for c0 in range(0, w.P, ce):
                    fa.fa_accumulate(silo, j, w.weights[k], fa.FA_KEY_FLAT, c0,
                                     bufs[k].data_ptr() + 2 * c0, min(ce, w.P - c0), sh)
            fa.fa_finalize(silo, [means[g]], sh)
        fa.fa_reset(top)
        ce32 = ce // 2                       # the same chunk bytes in fp32
        for g in range(S):
            for c0 in range(0, w.P, ce32):
                fa.fa_accumulate(top, g, totals[g], fa.FA_KEY_FLAT, c0,
                                 means[g].data_ptr() + 4 * c0, min(ce32, w.P - c0), sh)
        fa.fa_finalize(top, [out], sh)

    try:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        barrier(pg)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(args.steps):
            step()
        e1.record(s)
        torch.cuda.synchronize()
        ms = max_over_ranks(pg, e0.elapsed_time(e1) / args.steps)
    finally:
        fa.fa_close(silo)
        fa.fa_close(top)
    client_bytes = w.K * w.P * 2
    # silo streaming (first client 2 + 4, later 2 + 8 per element), silo finalize (4 + 4),
    # top level over fp32 means (first 4 + 4, later 4 + 8), top finalize (4 + 2)
    hbm = w.P * (S * (6 + 10 * (per - 1) + 8) + 8 + 12 * (S - 1) + 6)
    line = {"metric": METRIC, "mode": "hierarchical", "value": round(world * client_bytes / (ms * 1e-3) / 1e9, 2),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "P": w.P, "K": w.K, "silos": S, "clients_per_silo": per,
                       "silo_means": "fp32", "chunk_bytes": ce * 2},
            "hbm": {"bytes_per_round": int(hbm), "gbs": round(hbm / (ms * 1e-3) / 1e9, 1),
                    "frac": round(hbm / (ms * 1e-3) / 1e9 / peak, 4), "peak": peak,
                    "peak_kind": peak_kind}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-pool", type=int, default=24)
    ap.add_argument("--e2e-staged-steps", type=int, default=2,
                    help="also time the e2e round through the staging ring (0 = skip)")
    ap.add_argument("--ref-elems", type=int, default=64 << 20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-resident", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the rounds captured into a CUDA graph and replayed")
    ap.add_argument("--no-fused", action="store_true",
                    help="send the last client through fa_accumulate too (no fa_accumulate_final)")
    ap.add_argument("--no-compensated", action="store_true",
                    help="skip the round in the compensated mode (FA_COMPENSATED)")
    ap.add_argument("--ring-slots", type=int, default=0, help="e2e staging slots (0 = library default)")
    ap.add_argument("--slot-mb", type=int, default=0, help="e2e staging slot size in MiB (0 = default)")
    ap.add_argument("--hierarchical", type=int, default=0, metavar="S",
                    help="time a two-level round instead: S silos, then FedAvg over the silo means")
    ap.add_argument("--stage-host", action="store_true",
                    help="e2e: pinned chunks through the staging ring instead of read in place")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local, pg = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank, pg)
        if args.hierarchical > 0:
            return run_hierarchical(args, world, rank, local, pg)
        return run_ours(args, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
