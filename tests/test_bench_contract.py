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
    assert d["config"]["workload"].startswith("large:")
    import bench
    from combine_get_dispatch_gb300 import synth
    assert d["config"] == bench.config_of(synth.WORKLOADS["large"], 1)   # the GPU arm's config
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
    lrg = synth.WORKLOADS["large"]
    e2e = {"ms": 19.0, "serial_ms": 25.0, "h2d_bytes_per_step": 1891631104,
           "d2h_bytes_per_step": 1879048192}
    results = {
        "large": (lrg, SimpleNamespace(ll=False, rank=False),
                  measured(lrg, lrg.T * lrg.k, 1.63, 2.45, 4.13, e2e)),
        "decode": (dec, SimpleNamespace(ll=True, rank=False),
                   measured(dec, dec.T * dec.k, 0.032, 0.049, 0.081)),
    }
    args = bench.parse_args(["--steps", "20", "--warmup", "5"])
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    line = bench.assemble_line(args, 1, "large", results, clocks, 6750.0, "measured")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["value"] == pytest.approx(lrg.T / 4.13e-3) and line["ms_per_step"] == 4.13
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (1, 20, 5)
    assert line["config"]["workload"].startswith("large:") and "l2" in line["config"]
    rf = line["roofline"]
    assert rf["kernel"] == "k_combine" and rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["peak"] == 6750.0 and abs(rf["frac"] - rf["achieved"] / 6750.0) < 1e-3
    assert abs(rf["achieved"] - results["large"][2]["combine_gbs"]) < 0.1
    # the large combine moves 15.03 GB of rows in and 1.88 GB out per launch
    assert rf["alg_bytes_per_launch"] == lrg.T * lrg.k * 2 * lrg.H + lrg.T * 2 * lrg.H
    assert rf["traffic"] is None or rf["traffic"] > 0
    assert line["e2e"]["value"] == pytest.approx(lrg.T / 19.0e-3)
    assert line["e2e"]["h2d_bytes_per_step"] == 1891631104
    assert line["clocks"] == clocks and line["gpu_launches"] == 40
    assert set(line["workloads"]) == {"decode"}
    wd = line["workloads"]["decode"]
    assert wd["tokens_per_s"] == pytest.approx(dec.T / 0.081e-3)
    # every other workload carries its own roofline object
    rd = wd["roofline"]
    assert rd["kernel"] == "k_combine" and rd["frac"] == pytest.approx(
        results["decode"][2]["combine_gbs"] / 6750.0, abs=1e-3)


def test_traffic_key_ignores_comments_but_not_code(tmp_path):
    """The DRAM traffic the bench reports is keyed to a hash of the kernel
    source's code: a comment or whitespace edit keeps the key, a code edit
    changes it (and voids the stored traffic)."""
    import bench
    base = "// a kernel\n__global__ void k(int* p) {\n  p[0] = 1;   /* store */\n}\n"
    variants = {
        "comment": "// the same kernel, described differently\n__global__ void k(int* p) {\n  p[0] = 1;   /* one store */\n}\n",
        "spacing": "__global__   void k(int* p)\n{\n    p[0] = 1;\n}\n",
        "code": "// a kernel\n__global__ void k(int* p) {\n  p[0] = 2;   /* store */\n}\n",
    }
    src = tmp_path / "k.cu"
    src.write_text(base)
    key = bench.kernel_hash(str(src))
    for name, text in variants.items():
        src.write_text(text)
        assert (bench.kernel_hash(str(src)) == key) == (name != "code"), name
