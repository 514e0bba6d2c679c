"""The benchmark's reference arm (the CPU oracle timed on the host cores) and
its JSON line, on the 65 x 97 x 73 workload so that it runs in seconds.
No GPU: this arm never touches CUDA."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    return r


def test_reference_arm_line():
    r = run_bench("--impl", "reference", "--workload", "c1_bf16_65x97x73", "--steps", "2",
                  "--warmup", "1")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "bf16 GEMM+ReLU TFLOP/s at 65x97x73"
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["M"] == 65 and d["config"]["N"] == 97 and d["config"]["K"] == 73
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "D[0:65, 0:65]" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c1_bf16_65x97x73", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1",
                            "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rejects_batches():
    r = run_bench("--impl", "reference", "--workload", "c1_bf16_65x97x73", "--batch", "2")
    assert r.returncode != 0
    assert "unbatched" in r.stderr


def test_metric_names():
    sys.path.insert(0, ROOT)
    import bench
    import seeded_inputs as si

    assert bench.metric_name(si.WORKLOADS[bench.WORKLOAD]) == bench.METRIC
    assert bench.metric_name(si.WORKLOADS[bench.WORKLOAD], 1, "bf16") == \
        "bf16 GEMM+ReLU TFLOP/s at 8192x8192x8192, bf16 out"
    assert bench.metric_name(si.WORKLOADS["c3_fp16_4096"], 4, "bf16") == \
        "fp16 GEMM+ReLU TFLOP/s at 4096x4096x4096 x4, bf16 out"
    assert bench.metric_name(si.WORKLOADS["c2_tf32_256x128x512"]) == \
        "tf32 GEMM TFLOP/s at 256x128x512"
    assert bench.metric_name(si.WORKLOADS["mx_e2m1_8192"]).startswith(
        "block-scaled (32-element blocks) e2m1 GEMM+ReLU")


def test_input_copies_rule():
    """Inputs at least twice the L2 run as they are; smaller ones cycle
    through enough copies to reach that; tiny ones fall back to flushing."""
    sys.path.insert(0, ROOT)
    import bench
    import seeded_inputs as si

    l2 = bench.L2_BYTES
    assert bench.input_copies(2 * l2) == 1 and bench.input_copies(10 * l2) == 1
    assert bench.input_copies(2 * l2 - 1) == 2
    assert bench.input_copies(l2) == 2 and bench.input_copies(0.5 * l2) == 4
    assert bench.input_copies(2 * l2 / bench.MAX_COPIES) == bench.MAX_COPIES
    assert bench.input_copies(2 * l2 / bench.MAX_COPIES - 1e6) == 0
    assert bench.input_copies(0) == 0
    sizes = {n: bench.input_copies((w.M * w.K + w.K * w.N) * si.element_bytes(w.dtype))
             for n, w in si.WORKLOADS.items()}
    assert sizes["c4_bf16_8192"] == 1 and sizes["c3_fp16_4096"] == 4
    assert sizes["c5a_bf16_16384x64x4096"] == 2 and sizes["c5c_bf16_8191x4097x1000"] == 11
    assert sizes["c1_bf16_65x97x73"] == 0 and sizes["c2_tf32_256x128x512"] == 0


def test_roofline_bound_and_fractions():
    """The bound follows arithmetic intensity against the ridge of the given
    peaks; the 8-bit and 4-bit kinds scale the BF16 peak by the nominal
    ratios; algorithmic bytes count one scale byte per block."""
    sys.path.insert(0, ROOT)
    import bench
    import seeded_inputs as si

    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0, "hbm_gbs": 8000.0}
    c4 = si.WORKLOADS["c4_bf16_8192"]
    ms = c4.flops / 1000e12 * 1e3                   # exactly 1000 TFLOP/s
    r = bench.roofline(c4, ms, peaks, False)
    assert r["bound"] == "tensor" and abs(r["achieved"] - 1000.0) < 1e-6
    assert abs(r["frac"] - 0.5) < 1e-9 and r["peak"] == 2000.0
    assert bench.roofline(c4, ms, peaks, True)["peak"] == 1800.0
    c5a = si.WORKLOADS["c5a_bf16_16384x64x4096"]
    r = bench.roofline(c5a, 0.03, peaks, False)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 8000.0
    assert r["algorithmic_bytes_per_launch"] == (16384 * 4096 + 4096 * 64) * 2 + 16384 * 64 * 4
    f8 = si.WORKLOADS["f8_e4m3_8192"]
    assert bench.roofline(f8, 1.0, peaks, False)["peak"] == 4000.0
    nv = si.WORKLOADS["nvf4_8192"]
    r = bench.roofline(nv, 1.0, peaks, False)
    assert r["peak"] == 12000.0
    assert r["algorithmic_bytes_per_launch"] == \
        (2 * 8192 * 8192) * 0.5 + 8192 * 8192 * 4 + 2 * 8192 * (8192 // 16)
