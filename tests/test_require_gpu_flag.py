"""TG_REQUIRE_GPU turns the GPU tests' skips into failures where no device is
visible (run here in a child pytest with every GPU hidden)."""

import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TARGET = "tests/test_gpu_golden.py"


def run_child(require):
    env = {**os.environ, "CUDA_VISIBLE_DEVICES": ""}
    env.pop("TG_REQUIRE_GPU", None)
    if require is not None:
        env["TG_REQUIRE_GPU"] = require
    return subprocess.run([sys.executable, "-m", "pytest", TARGET, "-m", "gpu", "-q", "-x",
                           "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=300)


def test_gpu_tests_skip_without_the_flag():
    r = run_child(None)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "skipped" in r.stdout and "failed" not in r.stdout


def test_gpu_tests_fail_with_the_flag():
    r = run_child("1")
    assert r.returncode != 0
    assert "TG_REQUIRE_GPU is set but no CUDA device is visible" in r.stdout


def test_flag_zero_means_off():
    r = run_child("0")
    assert r.returncode == 0, r.stdout + r.stderr
