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


def test_roofline_kinds():
    """Tensor-bound workloads are placed against the bf16 peak, the grouped
    layer against HBM, ridge workloads on the larger of both fractions, the
    fp32 tensor-core path against the nominal 3xTF32 ceiling and the CUDA-core
    path against the FFMA rate."""
    sys.path.insert(0, ROOT)
    import bench
    from conv2d_backward_implicit_bwd_gb300 import workloads as wl
    peaks = {"source": "measured", "bf16_tflops": 2000.0, "hbm_gbs": 8000.0}
    big = wl.case("bf16_16x1x512x2048")
    r = bench.roofline_of("tcgen05", big, 2e12, 1e9, 1.0, peaks)  # 2 PFLOP/s, 1 TB/s
    assert r["bound"] == "tensor" and abs(r["frac"] - 1.0) < 1e-12 and abs(r["hbm_frac"] - 0.125) < 1e-12
    grp = wl.case("bf16_resnext")
    r = bench.roofline_of("grouped", grp, 2e9, 4e9, 1.0, peaks)
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-12
    ridge = wl.case("bf16_32x14x14_1024")
    r = bench.roofline_of("tcgen05", ridge, 2e11, 6e9, 1.0, peaks)  # tensor 0.1, hbm 0.75
    assert r["bound"] == "hbm" and r["frac"] == r["hbm_frac"] and r["graded_on"] == "max(tensor, hbm)"
    f32 = wl.case("fp32_nhwc_32x28x28x512")
    r = bench.roofline_of("tf32", f32, 1e11, 1e9, 1.0, peaks)
    assert abs(r["peak"] - 2000.0 * 1.1 / 2.25 / 3) < 1e-9 and "nominal" in r["peak_source"]
    small = wl.case("fp32_2x16x15x15")
    r = bench.roofline_of("simt", small, 1e9, 1e6, 1.0, peaks, sm_max_mhz=2000.0, num_sms=100)
    assert r["bound"] == "alu" and abs(r["peak"] - 100 * 128 * 2 * 2000e6 / 1e12) < 1e-9
