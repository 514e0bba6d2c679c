"""Batched GEMM and narrow (BF16/FP16) outputs through tg_gemm_batched,
against the oracle applied per batch entry plus its output rounding
("Matrix Multiplication", Step 4 and "Where to go from here")."""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import check_batched

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


@pytest.mark.parametrize("out", ["f32", "bf16", "fp16"])
@pytest.mark.parametrize("w", [
    si.Workload("pair", 600, 520, 1024, "bf16", 1.0, True, 81, "normal", scale=0.5, ldc=604),
    si.Workload("single", 300, 260, 200, "fp16", -0.5, False, 82, "uniform", lda=208, ldb=200),
    si.Workload("plain", 130, 70, 73, "bf16", 1.5, True, 83, "uniform"),
    si.Workload("tf32", 200, 150, 96, "tf32", 1.0, False, 84, "uniform", lo=0.0),
], ids=lambda w: w.name)
def test_batched_outputs(w, out):
    check_batched(w, 3, out, repeats=2)


def test_shared_operand_and_gaps():
    """stride_b = 0 (one B for all entries), padding between entries of A, B
    and D; the gaps of D stay untouched."""
    w = si.Workload("shared", 500, 300, 512, "bf16", 1.0, True, 85, "normal")
    check_batched(w, 4, "bf16", share_b=True, pad_a=64, pad_d=24)
    check_batched(w, 2, "f32", share_a=True, pad_b=8)


def test_swapped_vector_store_narrow():
    """Short M: roles swapped, 16-byte vector stores of BF16 output."""
    w = si.Workload("swapv", 40, 1000, 256, "bf16", 1.0, True, 86, "uniform", ldc=48)
    check_batched(w, 2, "bf16", pad_d=16)
    w2 = si.Workload("swaps", 40, 1000, 256, "fp16", 1.0, False, 87, "uniform", ldc=41)
    check_batched(w2, 2, "fp16", pad_d=3)


def test_batched_split_k():
    """Fewer pair tiles than pairs across the whole batch: K segments."""
    import dense_gemm_epilogue_gb300 as tg

    w = si.Workload("bsplit", 300, 256, 4096, "bf16", 1.0, True, 88, "normal")
    check_batched(w, 2, "fp16", repeats=2, opts={"cta_pair": 2, "block_n": 256})


def test_empty_and_zero_k():
    import torch
    import dense_gemm_epilogue_gb300 as tg

    D = torch.full((4 * 64,), 7.0, device="cuda")
    A = torch.zeros(64, dtype=torch.int16, device="cuda")
    assert tg.tg_gemm_batched(8, 8, 8, 1.0, A, 8, 0, A, 8, 0, D, 8, 64, 0, "bf16", "f32",
                              True) == tg.TG_OK
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)
    w = si.Workload("k0", 50, 40, 0, "fp16", -2.0, False, 89, "uniform", lda=1, ldb=1, ldc=52)
    check_batched(w, 3, "bf16", pad_d=8)


def test_invalid_batched_arguments():
    import torch
    import dense_gemm_epilogue_gb300 as tg

    D = torch.zeros(1000, device="cuda")
    A = torch.zeros(1000, dtype=torch.int16, device="cuda")
    bad = [
        dict(sd=8 * 8 - 1),   # outputs overlap
        dict(sa=-1), dict(sb=-2), dict(batch=-1), dict(out=3),
    ]
    for b in bad:
        a = dict(sa=64, sb=64, sd=64, batch=2, out=0)
        a.update(b)
        st = tg.tg_gemm_batched(8, 8, 8, 1.0, A, 8, a["sa"], A, 8, a["sb"], D, 8, a["sd"],
                                a["batch"], "bf16", a["out"], True)
        assert st == tg.TG_ERR_INVALID_VALUE, b
