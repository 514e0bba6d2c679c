"""Stream-K single-CTA tiles (option schedule = 3, and the planner's choice
for fewer tiles than SMs) against the oracle, every element, through the C
ABI: tiles cut between CTAs at every position (several cuts per tile, a
CTA's whole share inside one tile, shares spanning several tiles), every
operand kind and producer, batches, swapped roles, narrow outputs and a
composed epilogue; bitwise repeatable; the flags left clear for the next
launch."""

from __future__ import annotations

import pytest

import seeded_inputs as si
from gemm_harness import check_batched, check_epi, check_full

pytestmark = pytest.mark.gpu
SK = {"schedule": 3}


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


def _plan(w, opts):
    import dense_gemm_epilogue_gb300 as tg

    lda, ldb, ldc = w.strides
    return tg.tg_plan(w.M, w.N, w.K, None, lda, None, ldb, None, ldc, w.dtype, opts)


@pytest.mark.parametrize("block_n", [64, 128, 256])
@pytest.mark.parametrize("M,N,K", [(128, 64, 4096), (1000, 700, 3000), (300, 129, 1100)])
def test_stream_k_shapes(M, N, K, block_n):
    """One tile over 8 CTAs (7 partials into one owner), ragged tiles, K not a
    multiple of the stage."""
    w = si.Workload("sk", M, N, K, "bf16", 1.25, True, 700 + M + K, "normal", ldc=M + 3)
    opts = dict(SK, block_n=block_n)
    assert _plan(w, opts)["stream_k"] == 1
    check_full(w, opts=opts, repeats=3)


@pytest.mark.parametrize("ctas", [3, 7, 19])
def test_stream_k_shares_span_tiles(ctas):
    """More tiles than CTAs: each share crosses several tile boundaries and
    cuts tiles at both ends."""
    w = si.Workload("sk_span", 1100, 600, 1536, "fp16", -0.5, True, 710 + ctas, "uniform")
    opts = dict(SK, max_ctas=ctas, block_n=128)
    p = _plan(w, opts)
    assert p["stream_k"] == 1 and p["grid"] == ctas and p["tiles"] > ctas
    check_full(w, opts=opts, repeats=2)


@pytest.mark.parametrize("dtype", ["tf32", "e4m3", "e5m2"])
def test_stream_k_kinds(dtype):
    w = si.Workload("sk_kind", 333, 200, 2100, dtype, 1.0, False, 720, "normal")
    check_full(w, opts=SK, repeats=2)


def test_stream_k_plain_loads():
    """TMA-illegal strides: the plain-load producer walks the same units."""
    w = si.Workload("sk_plain", 257, 190, 1203, "bf16", 1.0, True, 730, "normal", lda=1205,
                    ldb=1207)
    opts = dict(SK, producer=2)
    assert _plan(w, opts)["producer"] == 2
    check_full(w, opts=opts, repeats=2)


def test_stream_k_swap_and_batches():
    w = si.Workload("sk_swap", 64, 2000, 2048, "bf16", 0.75, True, 740, "normal")
    check_full(w, opts=dict(SK, swap_ab=2), repeats=2)
    b = si.Workload("sk_batch", 300, 260, 1024, "fp16", 1.0, True, 745, "normal", ldc=304)
    check_batched(b, 3, "bf16", share_a=True, opts=SK, repeats=2)


def test_stream_k_composed_epilogue():
    w = si.Workload("sk_epi", 200, 300, 2048, "bf16", 1.0, False, 750, "normal")
    ops = [("bias_row", 0.0, 0.0, "rows"), ("silu", 0.0, 0.0, None), ("bias_col", 0.0, 0.0, "cols")]
    check_epi(w, ops, out="fp16", opts=SK, repeats=2)


@pytest.mark.parametrize("name", ["c5a_bf16_16384x64x4096", "c5b_bf16_64x16384x4096",
                                  "c2_tf32_256x128x512"])
def test_configs_under_stream_k(name):
    """The configurations' own shapes forced onto stream-K, and under the
    static schedule."""
    w = si.WORKLOADS[name]
    check_full(w, opts=SK, repeats=2)
    check_full(w, opts={"schedule": 1})


def test_long_k_planner_choice():
    """256 x 256 x 65536: the planner's stream-K over 152 CTAs (19 CTAs per
    tile, 18 partials summed by each owner)."""
    w = si.Workload("sk_long", 256, 256, 65536, "bf16", 1.0, True, 760, "uniform")
    p = _plan(w, None)
    assert p["stream_k"] == 1
    check_full(w, repeats=2)
