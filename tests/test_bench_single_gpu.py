"""The benchmark's GPU arm runs on exactly one GPU.  The library's CTA-pair
kernel can load A tiles with cluster-multicast TMA, which only single-GPU
calls may run, so there is no replica mode: asking for more than one GPU,
through --gpus or a multi-rank launch (WORLD_SIZE), must fail loudly before
any GPU work.  No GPU needed: the refusal comes first."""

import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(args, **env):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=300, cwd=ROOT,
                          env={**os.environ, "CUDA_VISIBLE_DEVICES": "", **env})


def test_gpus_two_is_refused():
    r = run_bench(["--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert r.returncode != 0
    assert "single-GPU library: replicas not run" in r.stderr
    assert r.stdout.strip() == ""


def test_world_size_two_is_refused_on_every_rank():
    for rank in ("0", "1"):
        r = run_bench(["--steps", "1", "--warmup", "0"], RANK=rank, LOCAL_RANK=rank,
                      WORLD_SIZE="2")
        assert r.returncode != 0, rank
        assert "WORLD_SIZE 2" in r.stderr
        assert r.stdout.strip() == ""


def test_refusal_rule():
    sys.path.insert(0, ROOT)
    import argparse

    import bench

    ok = argparse.Namespace(gpus=1)
    assert bench.single_gpu_refusal(ok, 1) is None
    assert bench.single_gpu_refusal(ok, 4) is not None
    assert bench.single_gpu_refusal(argparse.Namespace(gpus=8), 1) is not None
    assert bench.single_gpu_refusal(argparse.Namespace(gpus=0), 1) is not None
