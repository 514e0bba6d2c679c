"""tg_gemm_noalloc, the entry point for callers that cannot allocate device
memory: a process whose device memory is all held by its own pool
allocator, a latency-critical loop that must avoid cudaMalloc's implicit
synchronisation, or code running inside a stream capture that forbids
cudaMalloc.  Its kernel keeps its scratch (the status word of its bounded
waits) in a fixed array inside the library instead of memory the library
allocates, and it never splits K (that would need a workspace).

Checked through the C ABI:
- parity: every element against the oracle at the contract tolerance, on two
  calls in a row, with D's stride padding untouched; and against the
  allocating entry point, tg_gemm, on the same inputs within the same bound.
  The cases cover every planner branch: single-CTA TMA tiles, plain loads,
  swapped roles, a long K loop that tg_gemm splits and this call does not,
  CTA-pair tiles, two-pair multicast clusters, TF32, and the K = 0 fill with
  a negative alpha;
- empty outputs (M = 0, N = 0) launch nothing;
- bad arguments are rejected before anything is enqueued;
- in a fresh process without torch, calls after the set-up call leave the
  device's free memory unchanged, while the allocating entry point's
  workspace on the same stream is visible to the same measurement.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process.
"""

from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import (TOL_ABS, TOL_REL, assert_padding_untouched, assert_within, logical,
                          torch_storage)

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    # TMA producer, several tiles per CTA, ragged M/N/K, ReLU.
    si.Workload("noalloc_tma", 1000, 777, 300, "bf16", 1.5, True, 71, "uniform", ldc=1004),
    # Plain-load producer (TMA-illegal strides), the 65 x 97 x 73 example.
    si.WORKLOADS["c1_bf16_65x97x73"],
    # Roles swapped (short M), FP16, no epilogue, negative alpha.
    si.Workload("noalloc_swap", 40, 900, 200, "fp16", -0.5, False, 72, "normal", scale=0.1,
                ldc=44),
    # A long K loop that tg_gemm splits across CTA pairs; this call runs it unsplit.
    si.Workload("noalloc_unsplit", 600, 900, 2048, "bf16", 1.0, True, 74, "normal", ldc=600),
    # CTA-pair tiles.
    si.Workload("noalloc_pair", 1999, 1501, 1000, "bf16", 0.75, True, 76, "normal", ldc=2004),
    # Two CTA pairs per cluster sharing A rows by multicast (short K, many tiles).
    si.Workload("noalloc_multicast", 4000, 4900, 1000, "bf16", 1.0, True, 75, "uniform",
                lda=1008, ldb=1008, ldc=4004),
    # TF32 narrowing warps.
    si.Workload("noalloc_tf32", 300, 200, 96, "tf32", 1.0, False, 73, "uniform", lo=0.0),
    # K = 0: D = epi(alpha * 0); with alpha < 0 the ReLU turns -0 into +0.
    si.Workload("noalloc_k0_relu", 70, 90, 0, "bf16", -2.0, True, 1, "uniform", lda=1, ldb=1,
                ldc=72),
    si.Workload("noalloc_k0_plain", 70, 90, 0, "bf16", -2.0, False, 1, "uniform", lda=1, ldb=1,
                ldc=72),
]


@pytest.fixture(scope="module")
def tg():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()
    return tg


def _plan_branch(tg, w):
    lda, ldb, ldc = w.strides
    return tg.tg_plan(w.M, w.N, w.K, None, lda, None, ldb, None, ldc, w.dtype, {"split_k": 1})


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_oracle_twice(tg, w):
    import torch
    import oracle

    if w.name == "noalloc_multicast":
        assert _plan_branch(tg, w)["multicast"] == 2
    if w.name == "noalloc_pair":
        assert _plan_branch(tg, w)["cta_pair"] == 1
    if w.name == "noalloc_unsplit":
        lda, ldb, ldc = w.strides
        assert tg.tg_plan(w.M, w.N, w.K, None, lda, None, ldb, None, ldc, w.dtype)["split_segs"] > 1
        assert _plan_branch(tg, w)["split_segs"] == 1
    lda, ldb, ldc = w.strides
    A, B = si.make_operands(w)
    D0 = si.make_output(w)
    dA, dB = torch_storage(A), torch_storage(B)
    stream = torch.cuda.current_stream()
    ref, scale = oracle.gemm(w.M, w.N, w.K, w.alpha, A, lda, B, ldb, w.dtype, w.relu,
                             with_scale=True)

    # The allocating entry point on the same inputs.
    d_alloc = torch.from_numpy(D0.copy()).cuda()
    tg.check(tg.tg_gemm(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, d_alloc, ldc, w.dtype, w.relu,
                        stream))
    torch.cuda.synchronize()
    alloc_out = logical(d_alloc.cpu().numpy(), w).astype(np.float64)

    d_out = torch.from_numpy(D0.copy()).cuda()
    for call in range(2):
        st = tg.tg_gemm_noalloc(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, d_out, ldc, w.dtype,
                                w.relu, stream)
        assert st == tg.TG_OK, f"call {call}: {tg.tg_status_string(st)}"
        torch.cuda.synchronize()
        store = d_out.cpu().numpy()
        assert_padding_untouched(store, D0, w)
        got = logical(store, w)
        assert_within(got, ref, scale, w.dtype, f"{w.name} call {call} vs oracle")
        bound = TOL_REL[w.dtype] * scale + TOL_ABS
        assert np.all(np.abs(got.astype(np.float64) - alloc_out) <= bound), \
            f"{w.name} call {call}: differs from tg_gemm beyond the tolerance"
        if w.K == 0:
            # The empty sum exactly, sign of zero included (-0 without ReLU, +0 with it).
            want = ref.astype(np.float32)
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
            assert bool(np.signbit(got).all()) == (not w.relu)


def test_noalloc_empty_outputs_launch_nothing(tg):
    import torch

    D = torch.full((8, 8), 5.0, device="cuda")
    A = torch.zeros((8, 8), dtype=torch.int16, device="cuda")
    assert tg.tg_gemm_noalloc(0, 8, 8, 1.0, A, 8, A, 8, D, 8, "bf16", True) == tg.TG_OK
    assert tg.tg_gemm_noalloc(8, 0, 8, 1.0, A, 8, A, 8, D, 8, "bf16", True) == tg.TG_OK
    assert tg.tg_gemm_noalloc(0, 0, 0, 1.0, None, 1, None, 1, None, 1, "bf16", True) == tg.TG_OK
    torch.cuda.synchronize()
    assert torch.all(D == 5.0)


def test_noalloc_rejects_bad_arguments(tg):
    import torch

    D = torch.full((8, 8), 3.0, device="cuda")
    A = torch.zeros((8, 8), dtype=torch.int16, device="cuda")
    bad = [
        (8, 8, 8, A, 7, A, 8, D, 8, 0, 1),       # lda < K
        (8, 8, 8, None, 8, A, 8, D, 8, 0, 1),    # NULL A with M*K > 0
        (8, 8, 8, A, 8, A, 8, None, 8, 0, 1),    # NULL D
        (8, 8, 8, A, 8, A, 8, D, 8, 5, 1),       # bad dtype
        (8, 8, 8, A, 8, A, 8, D, 8, 0, 7),       # bad epilogue
    ]
    for M, N, K, a, la, b, lb, d, lc, dt, ep in bad:
        assert tg.tg_gemm_noalloc(M, N, K, 1.0, a, la, b, lb, d, lc, dt, ep) == \
            tg.TG_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert torch.all(D == 3.0)


def test_noalloc_allocates_nothing_after_setup(tg):
    """A fresh torch-free process: free device memory is unchanged across two
    passes of every case on a new stream, and the allocating entry point's
    workspace on that stream shows up in the same measurement."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "noalloc_probe.py")],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert d["free_after"] == d["free_before"], d
    assert d["control_split_segs"] > 1, d
    assert d["free_after"] - d["free_control"] >= 16 << 20, d
