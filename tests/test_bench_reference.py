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
