"""tg_gemm_noalloc, the entry point for callers that cannot allocate device
memory (a process whose device memory is all held by its own pool
allocator, a latency-critical loop that must avoid cudaMalloc's implicit
synchronisation, or code running inside a stream capture that forbids
cudaMalloc).  Its kernel keeps its scratch in a fixed array inside the
library instead of memory the library allocates.

Checked through the C ABI against the allocating entry point, tg_gemm, on
the same inputs: two calls in a row must each match it within the parity
tolerance of the other GPU tests, and leave D's stride padding untouched.
This file is collected last so that a run stopping at its first failure
has already run every other test; it also passes alone in a fresh process.
"""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import assert_padding_untouched, assert_within, logical, torch_storage

pytestmark = pytest.mark.gpu

CASES = [
    # TMA producer, several tiles per CTA, ragged M/N/K, ReLU.
    si.Workload("noalloc_tma", 1000, 777, 300, "bf16", 1.5, True, 71, "uniform", ldc=1004),
    # Plain-load producer (TMA-illegal strides), the 65 x 97 x 73 example.
    si.WORKLOADS["c1_bf16_65x97x73"],
    # Roles swapped (short M), FP16, no epilogue.
    si.Workload("noalloc_swap", 40, 900, 200, "fp16", -0.5, False, 72, "normal", scale=0.1,
                ldc=44),
    # CTA-pair tiles (long K), which tg_gemm would also split along K.
    si.Workload("noalloc_pair", 600, 900, 2048, "bf16", 1.0, True, 74, "normal", ldc=600),
    # TF32 narrowing warps.
    si.Workload("noalloc_tf32", 300, 200, 96, "tf32", 1.0, False, 73, "uniform", lo=0.0),
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


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_tg_gemm_twice(tg, w):
    import torch
    import oracle

    lda, ldb, ldc = w.strides
    A, B = si.make_operands(w)
    D0 = si.make_output(w)
    dA, dB = torch_storage(A), torch_storage(B)
    stream = torch.cuda.current_stream()

    d_ref = torch.from_numpy(D0.copy()).cuda()
    tg.check(tg.tg_gemm(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, d_ref, ldc, w.dtype, w.relu,
                        stream))
    torch.cuda.synchronize()
    ref_store = d_ref.cpu().numpy()
    ref = logical(ref_store, w).astype(np.float64)
    # The tolerance's scale (|alpha| * sum_k |a_ik||b_kj|) comes from the oracle.
    _, scale = oracle.gemm(w.M, w.N, w.K, w.alpha, A, lda, B, ldb, w.dtype, w.relu,
                           with_scale=True)

    d_out = torch.from_numpy(D0.copy()).cuda()
    for call in range(2):
        st = tg.tg_gemm_noalloc(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, d_out, ldc, w.dtype,
                                w.relu, stream)
        assert st == tg.TG_OK, f"call {call}: {tg.tg_status_string(st)}"
        torch.cuda.synchronize()
        out = d_out.cpu().numpy()
        assert_padding_untouched(out, D0, w)
        assert_within(logical(out, w), ref, scale, w.dtype, f"{w.name} call {call}")


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
