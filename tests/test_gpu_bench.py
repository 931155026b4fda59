"""bench.py end to end on the GPU, on the small tiny-CNN workload: one JSON line with
every key of the contract, byte counts that match the workload, and the reference
arm's line.  Runs bench.py as its own process, as the benchmark driver does."""
import json
import os
import subprocess
import sys

import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def test_bench_line_has_the_contract():
    w = W.make("tiny")
    si = 2 if w.dtype_in == "bf16" else 4
    so = 2 if w.dtype_out == "bf16" else 4
    d = _run("--workload", "tiny", "--steps", "2", "--warmup", "3", "--e2e-steps", "2",
             "--ref-elems", str(1 << 16))
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and d["dtype"] == "f32"
    assert d["config"]["workload"] == "tiny" and d["config"]["P"] == w.P and d["config"]["K"] == w.K
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # value = client bytes per step / time per step
    client = w.K * w.P * si
    assert abs(d["value"] - client / (d["ms_per_step"] * 1e-3) / 1e9) <= 0.05 * d["value"]   # rounding of ms
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["unit"] == "GB/s" and c["cores"] >= 1 and c["value"] > 0
    assert c["value_1thread"] > 0 and c["sample"]
    e = d["e2e"]
    assert e["unit"] == "GB/s" and e["value"] > 0
    assert e["h2d_bytes_per_step"] == client               # every client byte crosses the link
    assert e["d2h_bytes_per_step"] == w.P * so             # the aggregate comes back
    assert e["accumulate_ms"] > 0 and e["finalize_ms"] > 0 and e["h2d_peak_gbs"] > 0
    assert 0 < e["hbm_frac"] < 1 and e["hbm_gbs"] > 0
    # >= one accumulate per client per step (the last client's launches write the aggregate)
    assert d["gpu_launches"] >= 2 * w.K
    assert d["unfused"]["value"] > 0 and d["config"]["last_client"].startswith("fa_accumulate_final")
    assert d["resident"]["value"] > 0 and d["resident"]["launches_per_round"] >= 1
    # a small model's rounds, captured into CUDA graphs and replayed
    g = d["graph"]
    assert g["wall_ms_per_round"] > 0 and g["device_ms_per_round"] > 0 and g["calls_wall_ms_per_round"] > 0
    assert abs(g["value"] - client / (g["wall_ms_per_round"] * 1e-3) / 1e9) <= 0.05 * g["value"]
    assert d["resident"]["graph"]["wall_ms_per_round"] > 0
    assert d["delta_apply"]["gbs"] > 0 and d["delta_apply"]["bytes"] == w.P * (4 + 2 * so)
    cp = d["compensated"]
    assert cp["value"] > 0 and cp["bytes_per_round"] == w.P * (si + 8 + (w.K - 1) * (si + 16) + 8 + so)
    assert 0 < cp["accumulate"]["frac"] and cp["distinct_client_buffers"] >= 1
    assert 0 < d["partition_plan_us"] < 1000
    clk = d["clocks"]
    if clk is not None:
        assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk)


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
             "--ref-elems", str(1 << 16))
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_hierarchical_mode_line():
    from synth import workloads as W
    w = W.make("lora")
    d = _run("--workload", "lora", "--hierarchical", "2", "--steps", "2", "--warmup", "3")
    assert d["mode"] == "hierarchical" and d["config"]["silos"] == 2
    assert d["config"]["clients_per_silo"] == w.K // 2 and d["value"] > 0
    per = w.K // 2
    assert d["hbm"]["bytes_per_round"] == w.P * (2 * (6 + 10 * (per - 1) + 8) + 8 + 12 + 6)


def test_adapter_round_line():
    """The LoRA workload (clients send seeded subsets of the modules): the streamed round
    sends each client's reported keys only, and the `subsets` field times the one-pass
    round-level reduce over the same packed buffers."""
    import bench
    w = W.make("lora")
    d = _run("--workload", "lora", "--steps", "3", "--warmup", "3", "--e2e-steps", "2",
             "--no-cpu-baseline")
    cb = w.client_bytes()
    assert cb < w.K * w.P * 2                                # partial participation
    assert abs(d["value"] - cb / (d["ms_per_step"] * 1e-3) / 1e9) <= 0.05 * d["value"]
    sub = d["subsets"]
    assert sub["bytes_per_round"] == bench.subset_bytes(w) and sub["launches_per_round"] == 1
    assert sub["value"] > 0 and sub["hbm_frac"] > 0 and sub["wall_ms_per_round"] > 0
    assert d["resident"] is None and d["compensated"] is None
    assert d["e2e"]["h2d_bytes_per_step"] == cb
