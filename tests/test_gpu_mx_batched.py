"""Batched block-scaled GEMM with a composed epilogue, tg_gemm_mx_batched,
against the oracle's block-scaled product of each entry followed by its op
chain, element by element, through the C ABI: per-entry and shared operands
and scale sets, both 8-bit formats and packed FP4, narrow outputs, the role
swap, ragged tiles, K = 0 and batch = 0."""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import check_mx_batched

pytestmark = pytest.mark.gpu

CHAIN = [("bias_row", 0.0, 0.0, "rows"), ("gelu_tanh", 0.0, 0.0, None),
         ("bias_col", 0.0, 0.0, "cols"), ("clamp", -0.5, 2.0, None)]


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2", "e2m1", "nvf4"])
@pytest.mark.parametrize("M,N,K", [(300, 200, 320), (129, 65, 34), (257, 520, 1040)])
def test_mx_batched_per_entry(dtype, M, N, K):
    w = si.Workload(f"mxb_{dtype}", M, N, K, dtype, 1.25, False, 610 + M + K, "normal",
                    ldc=M + 5)
    check_mx_batched(w, 3, repeats=2)


@pytest.mark.parametrize("dtype", ["e4m3", "e2m1"])
def test_mx_batched_shared_operand_and_scales(dtype):
    """A and its scales shared by every entry; B per entry with one shared
    scale set; gaps between entries in every buffer."""
    w = si.Workload("mxb_share", 384, 300, 512, dtype, -0.5, False, 631, "uniform")
    check_mx_batched(w, 4, out="bf16", ops=[("relu", 0.0, 0.0, None)], share_a=True,
                     share_sfa=True, share_sfb=True, pad_b=64, pad_d=40)
    check_mx_batched(w, 3, out="f32", share_b=True, share_sfb=True, pad_a=32, pad_sf=48)


@pytest.mark.parametrize("dtype", ["e5m2", "e2m1"])
@pytest.mark.parametrize("out", ["f32", "bf16", "fp16"])
def test_mx_batched_chain(dtype, out):
    w = si.Workload("mxb_chain", 260, 390, 700 if dtype != "e2m1" else 704, dtype, 0.75, False,
                    640, "normal", ldc=264)
    check_mx_batched(w, 2, out=out, ops=CHAIN)


@pytest.mark.parametrize("swap", [1, 2])
@pytest.mark.parametrize("block_n", [128, 256])
def test_mx_batched_tile_configs_and_swap(swap, block_n):
    """Both tile widths with and without the role swap; the chain's row and
    column biases must follow D's rows and columns, not the kernel's roles."""
    w = si.Workload("mxb_cfg", 100, 700, 256, "e4m3", 1.0, False, 650, "normal")
    check_mx_batched(w, 3, ops=CHAIN, opts={"swap_ab": swap, "block_n": block_n})


@pytest.mark.parametrize("dtype", ["e4m3", "e2m1"])
def test_mx_batched_plain_loads(dtype):
    """Batch strides the TMA cannot address (A's entries 8 bytes off a
    16-byte boundary, B's odd rows): the plain-load producer, per-entry and
    shared scales."""
    ld = 522 if dtype == "e2m1" else 517
    w = si.Workload("mxb_plain", 260, 300, 512, dtype, 0.75, False, 670, "normal", lda=ld, ldb=ld)
    check_mx_batched(w, 3, ops=CHAIN, pad_a=16 if dtype == "e2m1" else 8, repeats=2)
    check_mx_batched(w, 3, out="bf16", share_b=True, share_sfb=True, pad_a=32, pad_sf=48)


def test_mx_batched_many_entries_persistent():
    """More tiles than CTA pairs: entries interleave across the persistent grid."""
    w = si.Workload("mxb_many", 512, 512, 256, "e4m3", 1.0, False, 660, "uniform")
    check_mx_batched(w, 24, out="bf16", ops=[("silu", 0.0, 0.0, None)], share_sfb=True,
                     opts={"max_ctas": 16})


def test_mx_batched_k_zero_and_empty_batch():
    """K = 0 writes out(ops(0)) into every entry without reading A, B or the
    scales; batch = 0 writes nothing."""
    import torch
    import dense_gemm_epilogue_gb300 as tg

    bias = torch.linspace(-1.0, 1.0, 30, device="cuda")
    D = torch.full((3, 20, 32), 7.0, device="cuda")
    ops = [("add", 0.25, 0.0, None), ("bias_row", 0.0, 0.0, bias)]
    st = tg.tg_gemm_mx_batched(30, 20, 0, 2.0, None, 16, 0, None, 0, None, 16, 0, None, 0, D, 32,
                               20 * 32, 3, "e4m3", "f32", ops)
    assert st == tg.TG_OK
    torch.cuda.synchronize()
    want = 0.25 + bias.cpu()
    got = D.cpu()
    for b in range(3):
        assert torch.equal(got[b, :, :30], want.expand(20, 30))
        assert torch.equal(got[b, :, 30:], torch.full((20, 2), 7.0))
    D2 = torch.full((20, 30), 7.0, device="cuda")
    st = tg.tg_gemm_mx_batched(30, 20, 64, 1.0, D2, 64, 0, D2, 0, D2, 64, 0, D2, 0, D2, 30, 600, 0,
                               "e4m3", "f32", ops)
    assert st == tg.TG_OK
    assert float(D2.min()) == 7.0 and float(D2.max()) == 7.0
