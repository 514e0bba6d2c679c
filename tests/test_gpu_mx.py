"""Block-scaled (microscaling) FP8 GEMM, tg_gemm_mx, against the oracle's
block-scaled product, element by element, through the C ABI; and the
scale-packing call against the layout's definition."""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import (check_mx, decode_out, logical, mx_padded, run_mx, to_atoms,
                          torch_storage)

pytestmark = pytest.mark.gpu
FP8 = ["e4m3", "e5m2"]


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


@pytest.mark.parametrize("rows,K,ld", [(1, 1, 1), (200, 283, 9), (128, 128, 4), (513, 4100, 140)])
def test_pack_scales_matches_layout(rows, K, ld):
    import dense_gemm_epilogue_gb300 as tg

    kb = (K + 31) // 32
    S = si.scale_codes(5, 2, rows, ld, 0, 254)
    dst = torch_storage(np.full(tg.tg_mx_scale_bytes(rows, K), 0xAB, dtype=np.uint8))
    tg.check(tg.tg_mx_pack_scales(rows, K, torch_storage(S), ld, dst), "tg_mx_pack_scales")
    got = dst.cpu().numpy()
    assert np.array_equal(got, to_atoms(S[:, :kb], K))


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (1, 1, 1), (129, 65, 33), (300, 520, 1040),
                                   (257, 255, 129), (513, 1000, 2048), (64, 1000, 512)])
def test_mx_shapes(dtype, M, N, K):
    w = si.Workload(f"mx_{dtype}", M, N, K, dtype, 1.5, True, 400 + M + N + K, "normal",
                    ldc=M + 3)
    check_mx(w, repeats=2)


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("swap", [1, 2])
def test_mx_tile_configs(dtype, block_n, swap):
    w = si.Workload("mx_cfg", 600, 700, 1000, dtype, -0.75, False, 91, "normal")
    check_mx(w, opts={"block_n": block_n, "swap_ab": swap})


@pytest.mark.parametrize("out", ["bf16", "fp16"])
def test_mx_narrow_outputs(out):
    """Narrow outputs; the wide scale range overflows FP16 in places (those
    elements must be the same infinities as the oracle's rounding)."""
    w = si.Workload("mx_out", 520, 600, 768, "e4m3", 0.5, True, 92, "normal")
    check_mx(w, out=out)
    check_mx(si.with_shape(w, seed=96, relu=False), out=out, scale_range=(122, 130))


def test_mx_persistent_and_wide_scale_range():
    """Few pairs (several tiles each, the single accumulator reused), and
    scales spanning 2^-40 .. 2^40."""
    w = si.Workload("mx_persist", 1100, 1300, 640, "e5m2", 1.0, True, 93, "normal")
    for g in (2, 6):
        check_mx(w, opts={"max_ctas": g, "raster_group": 2})
    check_mx(si.with_shape(w, seed=94), scale_range=(87, 167))


def test_mx_nan_scale_and_k_zero():
    import dense_gemm_epilogue_gb300 as tg
    import oracle

    w = mx_padded(si.Workload("mx_nan", 300, 200, 256, "e4m3", 1.0, True, 95, "normal"))
    A, B = si.make_operands(w)
    SA, SB = si.make_mx_scales(w)
    SA[17, 3] = 255
    SB[33, 0] = 255
    _, outs = run_mx(w, A, B, SA, SB)
    got = decode_out(outs[0][:, : w.M].view(np.float32).T, "f32")
    assert np.all(np.isnan(got[17])) and np.all(np.isnan(got[:, 33]))
    rest = np.delete(np.delete(got, 17, 0), 33, 1)
    assert not np.any(np.isnan(rest))
    lda, ldb, _ = w.strides
    ref = oracle.gemm_mx(w.M, w.N, w.K, w.alpha, A, lda, SA, 8, B, ldb, SB, 8, "e4m3", True)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    # K = 0: the epilogue of an empty sum, nothing read.
    import torch
    D = torch.full((20, 30), 7.0, device="cuda")
    st = tg.tg_gemm_mx(30, 20, 0, 2.0, None, 16, None, None, 16, None, D, 30, "e4m3", "f32",
                       False)
    assert st == tg.TG_OK
    assert float(D.abs().max()) == 0.0


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1, 1, 2), (129, 65, 34), (300, 520, 1040),
                                   (257, 255, 130), (513, 1000, 2048), (64, 1000, 512),
                                   (300, 200, 384), (130, 260, 130), (200, 300, 4000)])
def test_fp4_shapes(M, N, K):
    """Packed E2M1 with block scales: ragged edges; K = 384 and 130 leave an
    odd number of scale-atom columns (the last stage's second one is past
    the end and reads as zeros)."""
    w = si.Workload("mx_fp4", M, N, K, "e2m1", 1.5, True, 500 + M + N + K, "normal", ldc=M + 3)
    check_mx(w, repeats=2)


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("swap", [1, 2])
def test_fp4_tile_configs(block_n, swap):
    w = si.Workload("mx_fp4_cfg", 600, 700, 1024, "e2m1", -0.75, False, 97, "normal")
    check_mx(w, opts={"block_n": block_n, "swap_ab": swap})


def test_fp4_narrow_outputs_and_nan_scale():
    w = si.Workload("mx_fp4_out", 520, 600, 768, "e2m1", 0.5, True, 98, "normal")
    check_mx(w, out="bf16")
    check_mx(si.with_shape(w, seed=99, relu=False), out="fp16", scale_range=(122, 130))
    w = mx_padded(si.Workload("mx_fp4_nan", 300, 200, 256, "e2m1", 1.0, True, 95, "normal"))
    A, B = si.make_operands(w)
    SA, SB = si.make_mx_scales(w)
    SA[17, 3] = 255
    SB[33, 0] = 255
    _, outs = run_mx(w, A, B, SA, SB)
    got = decode_out(outs[0][:, : w.M].view(np.float32).T, "f32")
    assert np.all(np.isnan(got[17])) and np.all(np.isnan(got[:, 33]))
    assert not np.any(np.isnan(np.delete(np.delete(got, 17, 0), 33, 1)))


def _mx_plan(w, opts=None):
    import dense_gemm_epilogue_gb300 as tg

    lda, ldb, ldc = w.strides
    return tg.tg_plan_mx(w.M, w.N, w.K, lda, ldb, ldc, w.dtype, opts, 0)


@pytest.mark.parametrize("dtype,K,lda,ldb", [("e4m3", 1000, 1001, 1003), ("e5m2", 1000, 1000, 1024),
                                             ("e2m1", 1100, 1102, 1106), ("e2m1", 384, 400, 386)])
@pytest.mark.parametrize("block_n", [None, 256])
def test_mx_plain_loads(dtype, K, lda, ldb, block_n):
    """Row strides the TMA cannot address (odd byte strides included): the
    plain-load producer warps of both CTAs fill the stages and the scale
    atoms, ragged in every dimension; FP4 with K = 1100 and 384 leaves the
    last stage's second atom column past the end (read as zeros)."""
    w = si.Workload(f"mx_plain_{dtype}", 300, 390, K, dtype, 1.25, True, 530 + K + lda, "normal",
                    lda=lda, ldb=ldb, ldc=303)
    opts = {"block_n": block_n} if block_n else None
    plan = _mx_plan(w, opts)
    assert plan["producer"] == 2 and plan["block_n"] == (block_n or 128)
    check_mx(w, opts=opts, repeats=2)


@pytest.mark.parametrize("dtype", ["e4m3", "e2m1"])
def test_mx_plain_loads_swap_and_persistent(dtype):
    """Plain loads under the role swap, and with several tiles per pair."""
    lda = 514 if dtype == "e2m1" else 517
    w = si.Workload("mx_plain_swap", 64, 900, 512, dtype, -0.5, False, 541, "normal", lda=lda,
                    ldb=lda)
    assert _mx_plan(w)["producer"] == 2 and _mx_plan(w)["swap_ab"] == 1
    check_mx(w)
    w = si.Workload("mx_plain_persist", 1100, 700, 768, dtype, 1.0, True, 542, "uniform",
                    lda=lda + 256, ldb=lda + 258)
    check_mx(w, opts={"max_ctas": 6, "raster_group": 2})


@pytest.mark.parametrize("dtype", ["e4m3", "e2m1"])
def test_mx_plain_matches_tma(dtype):
    """Forcing the plain producer on TMA-legal operands gives the TMA
    producer's result bit for bit (the same stages, the same MMA order)."""
    w = mx_padded(si.Workload("mx_plain_same", 520, 600, 1024, dtype, 1.0, True, 543, "normal"))
    A, B = si.make_operands(w)
    SA, SB = si.make_mx_scales(w)
    _, tma = run_mx(w, A, B, SA, SB, opts={"producer": 1})
    _, plain = run_mx(w, A, B, SA, SB, opts={"producer": 2})
    assert np.array_equal(tma[0], plain[0])


@pytest.mark.parametrize("rows,K,ld", [(1, 2, 1), (200, 283, 18), (128, 64, 4), (513, 4100, 260)])
def test_nvf4_pack_scales_matches_layout(rows, K, ld):
    """16-element blocks: the block count and atom columns follow K / 16."""
    import dense_gemm_epilogue_gb300 as tg

    kb = (K + 15) // 16
    S = si.scale_codes(6, 2, rows, ld, 0, 0x7E)
    dst = torch_storage(np.full(tg.tg_bs_scale_bytes(rows, K, "nvf4"), 0xAB, dtype=np.uint8))
    tg.check(tg.tg_bs_pack_scales(rows, K, "nvf4", torch_storage(S), ld, dst), "tg_bs_pack_scales")
    assert np.array_equal(dst.cpu().numpy(), to_atoms(S[:, :kb], K, 16))


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1, 1, 2), (129, 65, 34), (300, 520, 1040),
                                   (257, 255, 130), (513, 1000, 2048), (64, 1000, 512),
                                   (300, 200, 18), (130, 260, 96), (200, 300, 4000)])
def test_nvf4_shapes(M, N, K):
    """NVFP4 (one unsigned-E4M3 scale per 16 K): ragged edges; K = 18, 34,
    96 and 130 end inside an atom column (later columns of the last stage
    read as zeros)."""
    w = si.Workload("nvf4", M, N, K, "nvf4", 1.5, True, 800 + M + N + K, "normal", ldc=M + 3)
    check_mx(w, repeats=2)


@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("swap", [1, 2])
def test_nvf4_tile_configs(block_n, swap):
    w = si.Workload("nvf4_cfg", 600, 700, 1024, "nvf4", -0.75, False, 801, "normal")
    check_mx(w, opts={"block_n": block_n, "swap_ab": swap})


def test_nvf4_scale_range_outputs_and_nan_scale():
    """Every finite scale code from the smallest subnormal to 448; narrow
    outputs; a NaN scale code (0x7F) makes its row or column NaN."""
    w = si.Workload("nvf4_out", 520, 600, 768, "nvf4", 0.5, True, 802, "normal")
    check_mx(w, scale_range=(0x01, 0x7E))
    check_mx(si.with_shape(w, seed=803, relu=False), out="bf16")
    check_mx(si.with_shape(w, seed=804), out="fp16", scale_range=(0x30, 0x40))
    w = mx_padded(si.Workload("nvf4_nan", 300, 200, 256, "nvf4", 1.0, True, 805, "normal"))
    A, B = si.make_operands(w)
    SA, SB = si.make_mx_scales(w)
    SA[17, 3] = 0x7F
    SB[33, 0] = 0x7F
    _, outs = run_mx(w, A, B, SA, SB)
    got = decode_out(outs[0][:, : w.M].view(np.float32).T, "f32")
    assert np.all(np.isnan(got[17])) and np.all(np.isnan(got[:, 33]))
    assert not np.any(np.isnan(np.delete(np.delete(got, 17, 0), 33, 1)))


def test_nvf4_plain_loads_and_persistent():
    """TMA-illegal rows (odd byte strides) on the plain-load producer, and
    several tiles per CTA pair."""
    w = si.Workload("nvf4_plain", 300, 390, 1100, "nvf4", 1.25, True, 806, "normal", lda=1102,
                    ldb=1106, ldc=303)
    assert _mx_plan(w)["producer"] == 2
    check_mx(w, repeats=2)
    w = si.Workload("nvf4_persist", 1100, 1300, 640, "nvf4", 1.0, True, 807, "normal")
    check_mx(w, opts={"max_ctas": 6, "raster_group": 2})


@pytest.mark.parametrize("name", ["mx_e4m3_8192", "mx_e2m1_8192", "nvf4_8192"])
def test_mx_8192_full(name):
    check_mx(si.WORKLOADS[name])
