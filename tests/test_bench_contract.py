"""The benchmark's reference arm (the CPU oracle, which needs no GPU) prints one
JSON line with the fields the benchmark contract asks of it, on the small fp32
workload so that the run takes seconds."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "fp32_2x16x15x15"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "dtype",
              "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 1 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["config"]["workload"] == "fp32_2x16x15x15_3x3_p1_s2"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_peaks_file_is_read_flat_or_nested(tmp_path):
    """The roofline denominators come from the measured-peaks file when it has
    the bf16 and HBM figures (at the top level or under a device entry), else
    from the stated fallback."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.load_peaks(str(tmp_path))["source"] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0}))
    p = bench.load_peaks(str(tmp_path))
    assert p["source"] == "measured" and p["hbm_gbs"] == 7000.0 and p["bf16_tflops"] == 2000.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"gpus": [{"index": 0, "hbm_gbs": 6900, "bf16_tflops": 1950, "bf16_tflops_sustained": 1700}]}))
    p = bench.load_peaks(str(tmp_path))
    assert p["source"] == "measured" and p["bf16_tflops_sustained"] == 1700.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0}))
    assert bench.load_peaks(str(tmp_path))["source"] == "fallback"
