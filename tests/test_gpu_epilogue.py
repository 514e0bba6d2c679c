"""Composed pointwise epilogues (tg_gemm_epilogue) against the oracle's
chain, element by element, through the C ABI: each op alone, chains with
row and column biases under both operand roles, every kernel family (single
CTA with TMA or plain loads, TF32, CTA pairs, 8-bit), narrow outputs and the
K = 0 path."""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import check_epi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


SINGLE_OPS = [("scale", -1.75, 0, None), ("add", 0.375, 0, None), ("relu", 0, 0, None),
              ("leaky_relu", 0.125, 0, None), ("clamp", -0.5, 1.25, None), ("sigmoid", 0, 0, None),
              ("silu", 0, 0, None), ("gelu_tanh", 0, 0, None), ("bias_row", 0, 0, "rows"),
              ("bias_col", 0, 0, "cols")]


@pytest.mark.parametrize("op", SINGLE_OPS, ids=lambda o: o[0])
def test_each_op(op):
    w = si.Workload("epi1", 300, 520, 200, "bf16", 1.5, False, 71, "normal", lda=208, ldb=216,
                    ldc=304)
    check_epi(w, [op])


CHAIN = [("scale", 0.5, 0, None), ("bias_col", 0, 0, "cols"), ("gelu_tanh", 0, 0, None),
         ("bias_row", 0, 0, "rows"), ("clamp", -1.0, 3.0, None), ("add", 0.125, 0, None)]


@pytest.mark.parametrize("swap", [1, 2])
@pytest.mark.parametrize("out", ["f32", "bf16", "fp16"])
def test_chain_both_roles(swap, out):
    """Row biases follow D's rows and column biases its columns whichever
    operand takes the MMA's M role."""
    w = si.Workload("epi_chain", 200, 333, 256, "fp16", -1.0, False, 72, "normal", ldc=205)
    check_epi(w, CHAIN, out=out, opts={"swap_ab": swap}, repeats=2)


@pytest.mark.parametrize("name,opts", [
    ("c1_bf16_65x97x73", None),                       # plain loads
    ("c2_tf32_256x128x512", None),                    # TF32 narrowing kernel
    ("pair", {"cta_pair": 2}),                        # CTA pairs
    ("mc", {"cta_pair": 2, "multicast": 2}),          # two-pair clusters
    ("split", {"cta_pair": 2, "max_ctas": 8, "split_k": 8}),  # split-K tail finisher
    ("fp8", None),
])
def test_kernel_families(name, opts):
    if name in si.WORKLOADS:
        w = si.WORKLOADS[name]
    elif name == "fp8":
        w = si.Workload("epi_fp8", 1100, 1300, 1024, "e4m3", 1.0, False, 73, "normal")
    elif name == "split":
        w = si.Workload("epi_split", 300, 600, 1024, "bf16", 1.0, False, 74, "normal")
    else:
        w = si.Workload("epi_pair", 1100, 1300, 640, "bf16", 1.0, False, 75, "normal")
    ops = [("bias_row", 0, 0, "rows"), ("silu", 0, 0, None), ("bias_col", 0, 0, "cols"),
           ("sigmoid", 0, 0, None)]
    check_epi(w, ops, opts=opts)


def test_k_zero_and_empty_chain():
    w = si.Workload("epi_k0", 70, 90, 0, "bf16", 2.0, True, 1, "uniform", lda=1, ldb=1, ldc=72)
    check_epi(w, [("add", 0.5, 0, None), ("bias_row", 0, 0, "rows"), ("bias_col", 0, 0, "cols")])
    w2 = si.Workload("epi_none", 130, 150, 96, "bf16", -0.5, False, 76, "normal")
    check_epi(w2, [])
