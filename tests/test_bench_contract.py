"""The benchmark's reference arm (the oracle timed on one host core) runs
without a GPU: its one JSON line must carry every field of the contract."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"].startswith("dispatch+combine tokens/s")
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and d["dtype"]
    assert d["config"]["workload"].startswith("decode:")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["unit"] == "tokens/s"
    assert cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}


def test_gpu_arm_line_from_measurements():
    """The GPU arm's line, assembled from stand-in measurements: every field
    the contract names, with value, roofline and end-to-end figures derived
    from them as stated."""
    from types import SimpleNamespace

    import bench
    from combine_get_dispatch_gb300 import synth

    def measured(w, rows, disp_ms, comb_ms, step_ms, e2e=None):
        st = {"median": step_ms * 1e3, "min": step_ms * 1e3, "p90": step_ms * 1e3}
        db, cb = bench.alg_bytes(w, rows)
        r = {"step_ms": step_ms, "step_ms_max": step_ms, "dispatch_ms": disp_ms,
             "combine_ms": comb_ms, "launches": 40, "step_us_stats": st,
             "dispatch_us_stats": st, "combine_us_stats": st, "dispatch_alg_bytes": db,
             "combine_alg_bytes": cb, "dispatch_gbs": db / (disp_ms * 1e-3) / 1e9,
             "combine_gbs": cb / (comb_ms * 1e-3) / 1e9, "tokens": w.T}
        if e2e:
            r["e2e"] = e2e
        return r

    dec = synth.WORKLOADS["decode"]
    pre = synth.WORKLOADS["prefill"]
    e2e = {"ms": 0.2, "serial_ms": 0.34, "h2d_bytes_per_step": 29556736,
           "d2h_bytes_per_step": 29360128}
    results = {
        "decode": (dec, SimpleNamespace(ll=True, rank=False),
                   measured(dec, dec.T * dec.k, 0.032, 0.049, 0.081, e2e)),
        "prefill": (pre, SimpleNamespace(ll=False, rank=False),
                    measured(pre, pre.T * pre.k, 0.73, 0.62, 1.37)),
    }
    args = bench.parse_args(["--steps", "20", "--warmup", "5"])
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    line = bench.assemble_line(args, 1, "decode", results, clocks, 6750.0, "measured")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["value"] == pytest.approx(dec.T / 0.081e-3) and line["ms_per_step"] == 0.081
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (1, 20, 5)
    assert line["config"]["workload"].startswith("decode:") and "l2" in line["config"]
    rf = line["roofline"]
    assert rf["kernel"] == "k_combine" and rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["peak"] == 6750.0 and abs(rf["frac"] - rf["achieved"] / 6750.0) < 1e-3
    assert abs(rf["achieved"] - results["decode"][2]["combine_gbs"]) < 0.1
    assert rf["traffic"] is None or rf["traffic"] > 0
    assert line["e2e"]["value"] == pytest.approx(dec.T / 0.2e-3)
    assert line["e2e"]["h2d_bytes_per_step"] == 29556736
    assert line["clocks"] == clocks and line["gpu_launches"] == 40
    assert set(line["workloads"]) == {"prefill"}
    assert line["workloads"]["prefill"]["tokens_per_s"] == pytest.approx(pre.T / 1.37e-3)
