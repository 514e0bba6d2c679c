"""The C-ABI library on the host (no GPU): it builds, loads, exports every
symbol the header declares, validates arguments before touching CUDA, and
its planner makes the documented choices."""

from __future__ import annotations

import os
import re
import subprocess

import pytest

import seeded_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tg_gemm.h")


@pytest.fixture(scope="module")
def tg():
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()
    return tg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names(tg):
    assert declared_functions() == sorted(tg.EXPORTED)


def test_library_exports_every_declared_symbol(tg):
    lib = tg.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", tg.LIBRARY_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (tg_[a-z0-9_]+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported


def test_status_strings_and_version(tg):
    assert tg.tg_status_string(0) == "TG_OK"
    assert tg.tg_status_string(4) == "TG_ERR_DEVICE_TIMEOUT"
    assert tg.tg_status_string(99) == "TG_ERR_UNKNOWN"
    assert tg.tg_version() == 100
    assert tg.tg_set_wait_limit_ns(0) == tg.TG_OK


FAKE = 1 << 20  # a 16-byte aligned non-NULL address; never dereferenced here


@pytest.mark.parametrize("args", [
    dict(M=-1), dict(N=-1), dict(K=-1),
    dict(lda=9), dict(ldb=9), dict(ldc=9),
    dict(A=None), dict(B=None), dict(D=None),
    dict(A=FAKE + 1), dict(D=FAKE + 2),
    dict(dtype=5), dict(dtype=-1), dict(epi=2),
    dict(opts={"block_n": 96}), dict(opts={"producer": 3}), dict(opts={"swap_ab": 3}),
    dict(opts={"raster_group": -1}), dict(opts={"max_ctas": -2}), dict(opts={"l2_hint": 3}),
    dict(opts={"split_k": -1}), dict(opts={"split_k": 65}), dict(opts={"prefetch_k": -2}),
    dict(opts={"reserved": [1]}), dict(opts={"multicast": 3}), dict(opts={"schedule": 5}),
    dict(opts={"schedule": 4, "cta_pair": 1}), dict(opts={"schedule": 4, "multicast": 2}),
    dict(opts={"schedule": 4, "split_k": 1}),
    dict(opts={"schedule": 3, "cta_pair": 2}), dict(opts={"schedule": 3, "split_k": 1}),
    dict(opts={"schedule": 3, "multicast": 2}),
    dict(opts={"schedule": 2, "cta_pair": 1}), dict(opts={"schedule": 2, "multicast": 2}),
    dict(opts={"schedule": 2, "split_k": 2}),
    dict(opts={"multicast": 2, "cta_pair": 1}),
    dict(opts={"cta_pair": 3}), dict(opts={"cta_pair": 2, "block_n": 64}),
    dict(dtype=2, opts={"cta_pair": 2}),
])
def test_invalid_arguments_rejected_before_cuda(tg, args):
    a = dict(M=10, N=10, K=10, A=FAKE, lda=10, B=FAKE, ldb=10, D=FAKE, ldc=10, dtype=0, epi=1,
             opts=None)
    a.update(args)
    st = tg.tg_gemm_ex(a["M"], a["N"], a["K"], 1.0, a["A"], a["lda"], a["B"], a["ldb"], a["D"],
                       a["ldc"], a["dtype"], a["epi"], a["opts"])
    assert st == tg.TG_ERR_INVALID_VALUE


def test_empty_output_is_ok_without_cuda(tg):
    assert tg.tg_gemm(0, 10, 10, 1.0, None, 10, FAKE, 10, None, 1, "bf16", True) == tg.TG_OK
    assert tg.tg_gemm(10, 0, 10, 1.0, FAKE, 10, None, 10, None, 10, "bf16", True) == tg.TG_OK


def test_tf32_alignment_is_element_size(tg):
    st = tg.tg_gemm(4, 4, 4, 1.0, FAKE + 2, 4, FAKE, 4, FAKE, 4, "tf32", False)
    assert st == tg.TG_ERR_INVALID_VALUE


def plan(tg, w, opts=None, sms=152, A=FAKE, B=FAKE, D=FAKE):
    lda, ldb, ldc = w.strides
    return tg.tg_plan(w.M, w.N, w.K, A, lda, B, ldb, D, ldc, w.dtype, opts, sms)


def test_plan_headline_8192(tg):
    p = plan(tg, si.WORKLOADS["c4_bf16_8192"])
    assert p["cta_pair"] == 1                       # 256 x 256 tiles over CTA pairs
    assert (p["block_m"], p["block_n"], p["block_k"]) == (256, 256, 64)
    assert p["producer"] == 1 and p["swap_ab"] == 0
    assert p["tiles"] == 32 * 32 and p["grid"] == 152
    assert p["stages"] == 7 and p["tmem_cols"] == 512 and p["threads"] == 320
    assert p["smem_bytes"] <= 232448
    s = plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"cta_pair": 1})
    assert (s["cta_pair"], s["block_m"], s["block_n"], s["tiles"]) == (0, 128, 256, 2048)
    assert s["stages"] == 4


def test_plan_split_tail(tg):
    """K segments for pair tiles: up to 8 when there are fewer tiles than
    pairs; with the ticket schedule (the default for a wave or more of pair
    tiles) the last partial wave is cut into two segments when at most half
    full; forced, the last partial wave (R = tiles mod pairs tiles) is cut
    into S = min(pairs // R, split_k, K blocks // 8) segments."""
    c4 = plan(tg, si.WORKLOADS["c4_bf16_8192"])        # 1024 tiles on 76 pairs
    assert (c4["split_tiles"], c4["split_segs"], c4["schedule"]) == (1024 % 76, 2, 4)
    static = plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"schedule": 1})
    assert (static["split_tiles"], static["split_segs"], static["schedule"]) == (36, 2, 1)
    # A last wave more than half full is not split (two segments would not fit).
    w = si.Workload("s", 256 * 12, 256 * 10, 4096, "bf16", 1.0, True, 0, "normal")
    more = plan(tg, w)                                   # 120 tiles: 44 in the last wave
    assert (more["split_segs"], more["schedule"]) == (1, 1)
    # No workspace, no tickets.
    nows = plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"split_k": 1})
    assert (nows["split_segs"], nows["schedule"]) == (1, 1)
    forced = plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"split_k": 8})
    assert (forced["split_tiles"], forced["split_segs"]) == (1024 % 76, 2)
    small = plan(tg, si.Workload("s", 500, 500, 2048, "bf16", 1.0, True, 0, "normal"),
                 opts={"cta_pair": 2, "block_n": 256})
    assert small["cta_pair"] == 1 and small["tiles"] == 4
    assert (small["split_tiles"], small["split_segs"]) == (4, 4)   # 32 K blocks / 8
    short_k = plan(tg, si.Workload("s", 500, 500, 512, "bf16", 1.0, True, 0, "normal"),
                   opts={"cta_pair": 2})
    assert short_k["split_segs"] == 1                            # 8 K blocks: no split
    single = plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"cta_pair": 1, "split_k": 8})
    assert (single["split_tiles"], single["split_segs"]) == (0, 1)


def test_plan_pair_needs_some_k(tg):
    c5c = plan(tg, si.WORKLOADS["c5c_bf16_8191x4097x1000"])      # 16 K blocks
    assert c5c["cta_pair"] == 1
    short = si.Workload("s", 4096, 4096, 256, "bf16", 1.0, True, 0, "normal")   # 4 K blocks
    assert plan(tg, short)["cta_pair"] == 0
    assert plan(tg, short, opts={"cta_pair": 2})["cta_pair"] == 1


def test_plan_tma_illegal_strides_use_plain_loads(tg):
    p = plan(tg, si.WORKLOADS["c1_bf16_65x97x73"])   # 73 * 2 bytes is not a multiple of 16
    assert p["producer"] == 2 and p["swap_ab"] == 0
    assert p["threads"] == 320 + 128                  # plus 4 loader warps
    with pytest.raises(tg.TgError):
        plan(tg, si.WORKLOADS["c1_bf16_65x97x73"], opts={"producer": 1})
    # A misaligned base also rules TMA out.
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"], A=FAKE + 2)["producer"] == 2


def test_plan_skinny_shapes(tg):
    a = plan(tg, si.WORKLOADS["c5a_bf16_16384x64x4096"])
    assert a["swap_ab"] == 0 and a["block_n"] == 64 and a["tiles"] == 128 and a["producer"] == 1
    b = plan(tg, si.WORKLOADS["c5b_bf16_64x16384x4096"])
    assert b["swap_ab"] == 1 and b["block_n"] == 64 and b["tiles"] == 128
    assert b["vector_store"] == 1                      # ldc = 72 keeps rows 16-byte aligned
    c = plan(tg, si.WORKLOADS["c5c_bf16_8191x4097x1000"])
    assert c["producer"] == 1 and c["swap_ab"] == 0


def test_plan_tf32(tg):
    p = plan(tg, si.WORKLOADS["c2_tf32_256x128x512"])
    assert p["block_k"] == 32 and p["threads"] == 448 and p["cta_pair"] == 0
    with pytest.raises(tg.TgError):
        plan(tg, si.WORKLOADS["c2_tf32_256x128x512"], opts={"cta_pair": 2})


def test_plan_fp8(tg):
    """8-bit floats: 128 K elements per stage (one 128-byte row), pair tiles
    from 8 K blocks on, TMA when strides are multiples of 16 bytes."""
    for dt in ("e4m3", "e5m2"):
        p = plan(tg, si.WORKLOADS[f"f8_{dt}_8192"])
        assert (p["block_m"], p["block_n"], p["block_k"]) == (256, 256, 128)
        assert p["cta_pair"] == 1 and p["producer"] == 1 and p["stages"] == 7
        assert p["tiles"] == 1024 and p["threads"] == 320
        assert plan(tg, si.Workload("s", 4096, 4096, 1024, dt, 1.0, True, 0, "normal"))["cta_pair"] == 1
        assert plan(tg, si.Workload("s", 4096, 4096, 896, dt, 1.0, True, 0, "normal"))["cta_pair"] == 0
        # lda = 1000 bytes: not a multiple of 16 -> plain loads; 1008 is.
        w = si.Workload("s", 300, 300, 1000, dt, 1.0, True, 0, "normal")
        assert plan(tg, w)["producer"] == 2
        assert plan(tg, si.with_shape(w, lda=1008, ldb=1008))["producer"] == 1
        # Any base address is element-aligned for 1-byte types.
        assert plan(tg, si.with_shape(w, lda=1008, ldb=1008), A=FAKE + 1)["producer"] == 2
        split = plan(tg, si.Workload("s", 500, 500, 8192, dt, 1.0, True, 0, "normal"),
                     opts={"cta_pair": 2})
        assert split["split_tiles"] == split["tiles"] and split["split_segs"] == 8  # 64 K blocks / 8


def test_plan_pair_grid_is_even_and_capped(tg):
    w = si.WORKLOADS["c3_fp16_4096"]
    p = plan(tg, w)
    assert p["cta_pair"] == 1 and p["block_m"] == 256 and p["grid"] % 2 == 0
    q = plan(tg, w, opts={"cta_pair": 2, "max_ctas": 7})
    assert q["grid"] == 6
    r = plan(tg, si.Workload("tiny", 200, 100, 64, "bf16", 1.0, True, 0, "uniform"),
             opts={"cta_pair": 2})
    assert r["tiles"] == 1 and r["grid"] == 2


def test_plan_overrides(tg):
    w = si.WORKLOADS["c3_fp16_4096"]
    p = plan(tg, w, opts={"block_n": 128, "max_ctas": 10, "raster_group": 4, "swap_ab": 2,
                          "cta_pair": 1})
    assert p["block_n"] == 128 and p["grid"] == 10 and p["raster_group"] == 4 and p["swap_ab"] == 1
    p = plan(tg, w, opts={"raster_group": 1000, "cta_pair": 1})
    assert p["raster_group"] == 32                     # clamped to the M tile count
    p = plan(tg, w, opts={"raster_group": 1000, "cta_pair": 2})
    assert p["raster_group"] == 16                     # 256-row tiles
    # 8 M tiles per group for pair tiles; 12 under the alternating K order.
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"])["raster_group"] == 12
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"schedule": 1})["raster_group"] == 8
    assert plan(tg, si.WORKLOADS["c3_fp16_4096"])["raster_group"] == 8
    assert plan(tg, w, sms=7, opts={"cta_pair": 1})["grid"] == 7
    assert plan(tg, w, sms=7)["grid"] == 6             # pairs: 3 clusters of 2


@pytest.mark.parametrize("args", [
    dict(sd=63), dict(sa=-1), dict(sb=-1), dict(batch=-1), dict(out=3), dict(D=FAKE + 1, out=1),
    dict(D=FAKE + 2, out=0), dict(dtype=2, opts={"cta_pair": 2}),
])
def test_batched_invalid_arguments_rejected_before_cuda(tg, args):
    a = dict(M=8, N=8, K=8, A=FAKE, lda=8, sa=64, B=FAKE, ldb=8, sb=64, D=FAKE, ldc=8, sd=64,
             batch=2, dtype=0, out=0, opts=None)
    a.update(args)
    st = tg.tg_gemm_batched(a["M"], a["N"], a["K"], 1.0, a["A"], a["lda"], a["sa"], a["B"], a["ldb"],
                            a["sb"], a["D"], a["ldc"], a["sd"], a["batch"], a["dtype"], a["out"], True,
                            a["opts"])
    assert st == tg.TG_ERR_INVALID_VALUE


def test_batched_empty_is_ok_without_cuda(tg):
    assert tg.tg_gemm_batched(8, 8, 8, 1.0, FAKE, 8, 64, FAKE, 8, 64, FAKE, 8, 64, 0, "bf16", "bf16",
                              True) == tg.TG_OK


def test_plan_multicast_clusters(tg):
    """Two CTA pairs per cluster share their A rows: a cluster covers two N
    blocks, the grid is a multiple of four CTAs, and no K split is used."""
    w = si.WORKLOADS["c4_bf16_8192"]
    one = plan(tg, w, opts={"multicast": 1})
    two = plan(tg, w, opts={"multicast": 2})
    assert one["multicast"] == 1 and two["multicast"] == 2
    assert two["tiles"] * 2 == one["tiles"] and two["grid"] % 4 == 0 and two["grid"] == 152
    assert two["split_segs"] == 1
    assert plan(tg, w, opts={"cta_pair": 1})["multicast"] == 0
    # The planner's own choice: short K loops over several waves share A rows.
    c5c = plan(tg, si.WORKLOADS["c5c_bf16_8191x4097x1000"])
    assert c5c["cta_pair"] == 1 and c5c["multicast"] == 2 and c5c["grid"] % 4 == 0
    assert plan(tg, si.WORKLOADS["c5c_bf16_8191x4097x1000"], opts={"multicast": 1})["multicast"] == 1
    assert plan(tg, w)["multicast"] == 1                                   # 128 K blocks
    assert plan(tg, si.WORKLOADS["c3_fp16_4096"])["multicast"] == 1        # 64 K blocks
    # A single N block leaves nothing to share.
    narrow = si.Workload("n", 4096, 200, 4096, "bf16", 1.0, True, 0, "normal")
    with pytest.raises(tg.TgError):
        plan(tg, narrow, opts={"multicast": 2, "cta_pair": 2, "block_n": 256})



# ----------------------------------------------------------------- block-scaled path (host only)

def test_mx_scale_bytes(tg):
    assert tg.tg_mx_scale_bytes(0, 100) == 0 and tg.tg_mx_scale_bytes(100, 0) == 0
    assert tg.tg_mx_scale_bytes(1, 1) == 512
    assert tg.tg_mx_scale_bytes(128, 128) == 512
    assert tg.tg_mx_scale_bytes(129, 129) == 4 * 512
    assert tg.tg_mx_scale_bytes(8192, 8192) == 64 * 64 * 512
    assert tg.tg_mx_scale_bytes(-1, 5) == -1


def test_bs_scale_bytes(tg):
    """Atoms of 128 rows x 4 blocks: 32-K blocks for the exponent-scaled
    types, 16-K blocks for nvf4 (twice the atom columns)."""
    for dt in ("e4m3", "e5m2", "e2m1"):
        assert tg.tg_bs_scale_bytes(129, 129, dt) == tg.tg_mx_scale_bytes(129, 129) == 4 * 512
    assert tg.tg_bs_scale_bytes(128, 64, "nvf4") == 512
    assert tg.tg_bs_scale_bytes(128, 65, "nvf4") == 2 * 512
    assert tg.tg_bs_scale_bytes(129, 129, "nvf4") == 2 * 3 * 512
    assert tg.tg_bs_scale_bytes(8192, 8192, "nvf4") == 64 * 128 * 512
    assert tg.tg_bs_scale_bytes(0, 100, "nvf4") == 0 and tg.tg_bs_scale_bytes(5, -1, "nvf4") == -1
    for dt in ("bf16", "fp16", "tf32", 7):
        assert tg.tg_bs_scale_bytes(10, 10, dt) == -1
    assert tg.tg_bs_pack_scales(10, 64, "bf16", FAKE, 4, FAKE) == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_bs_pack_scales(10, 64, "nvf4", FAKE, 3, FAKE) == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_bs_pack_scales(0, 64, "nvf4", None, 4, None) == tg.TG_OK


@pytest.mark.parametrize("args", [
    dict(K=1023, lda=1024, ldb=1024), dict(lda=1025, ldb=1025),
    dict(lda=1040, opts={"producer": 1}), dict(opts={"block_n": 64}),
])
def test_nvf4_layout_rules(tg, args):
    """NVFP4 takes the packed-FP4 rules: even K, lda, ldb; and only the
    block-scaled entry points."""
    a = dict(M=10, N=10, K=1024, lda=1024, ldb=1024, opts=None)
    a.update(args)
    st = tg.tg_gemm_mx(a["M"], a["N"], a["K"], 1.0, FAKE, a["lda"], FAKE, FAKE, a["ldb"], FAKE,
                       FAKE, 10, "nvf4", "f32", 1, a["opts"])
    assert st == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_gemm(10, 10, 64, 1.0, FAKE, 64, FAKE, 64, FAKE, 10, "nvf4", True) == \
        tg.TG_ERR_INVALID_VALUE
    p = tg.tg_plan_mx(8192, 8192, 8192, 8192, 8192, 8192, "nvf4", None, 152)
    assert (p["block_k"], p["tmem_cols"], p["cta_pair"]) == (256, 512, 1)
    assert p["block_n"] in (128, 256) and p["stages"] >= 5


@pytest.mark.parametrize("args", [
    dict(dtype="bf16"), dict(dtype="tf32"), dict(lda=1000), dict(ldb=1000),
    dict(A=FAKE + 8, opts={"producer": 1}), dict(lda=1032, opts={"producer": 1}),
    dict(SFA=None), dict(SFB=FAKE + 4), dict(epi=2), dict(out=3), dict(ldc=9),
    dict(opts={"block_n": 64}), dict(opts={"cta_pair": 1}), dict(opts={"split_k": 2}),
    dict(opts={"multicast": 2}), dict(opts={"producer": 3}), dict(opts={"l2_hint": 1}),
])
def test_mx_invalid_arguments_rejected_before_cuda(tg, args):
    a = dict(M=10, N=10, K=1024, A=FAKE, lda=1024, SFA=FAKE, B=FAKE, ldb=1024, SFB=FAKE, D=FAKE,
             ldc=10, dtype="e4m3", out="f32", epi=1, opts=None)
    a.update(args)
    st = tg.tg_gemm_mx(a["M"], a["N"], a["K"], 1.0, a["A"], a["lda"], a["SFA"], a["B"], a["ldb"],
                       a["SFB"], a["D"], a["ldc"], a["dtype"], a["out"], a["epi"], a["opts"])
    assert st == tg.TG_ERR_INVALID_VALUE


@pytest.mark.parametrize("args", [
    dict(lda=1025, ldb=1025), dict(K=1023, lda=1024, ldb=1024),
    dict(lda=1040, opts={"producer": 1}), dict(ldb=1040, opts={"producer": 1}),
])
def test_mx_fp4_layout_rules(tg, args):
    """Packed FP4: even lda, ldb and K; the TMA producer, when forced, wants
    row strides of 16-byte multiples."""
    a = dict(M=10, N=10, K=1024, lda=1024, ldb=1024, opts=None)
    a.update(args)
    st = tg.tg_gemm_mx(a["M"], a["N"], a["K"], 1.0, FAKE, a["lda"], FAKE, FAKE, a["ldb"], FAKE,
                       FAKE, 10, "e2m1", "f32", 1, a["opts"])
    assert st == tg.TG_ERR_INVALID_VALUE
    # Only the block-scaled path takes FP4.
    assert tg.tg_gemm(10, 10, 64, 1.0, FAKE, 64, FAKE, 64, FAKE, 10, "e2m1", True) == \
        tg.TG_ERR_INVALID_VALUE
    p = tg.tg_plan_mx(8192, 8192, 8192, 8192, 8192, 8192, "e2m1", None, 152)
    assert (p["block_k"], p["stages"], p["tmem_cols"]) == (256, 6, 512)


def test_mx_empty_output_is_ok_without_cuda(tg):
    assert tg.tg_gemm_mx(0, 10, 64, 1.0, None, 64, None, FAKE, 64, FAKE, None, 1, "e4m3", "f32",
                         True) == tg.TG_OK


def test_plan_mx(tg):
    p = tg.tg_plan_mx(8192, 8192, 8192, 8192, 8192, 8192, "e4m3", None, 152)
    assert (p["block_m"], p["block_n"], p["block_k"]) == (256, 256, 128)
    assert p["cta_pair"] == 1 and p["tiles"] == 1024 and p["grid"] == 152
    assert p["stages"] == 6 and p["tmem_cols"] == 512 and p["threads"] == 320
    assert p["smem_bytes"] <= 232448
    q = tg.tg_plan_mx(8192, 8192, 8192, 8192, 8192, 8192, "e5m2", {"block_n": 128}, 152)
    assert q["block_n"] == 128 and q["stages"] == 8 and q["tmem_cols"] == 256
    s = tg.tg_plan_mx(64, 4096, 1024, 1024, 1024, 64, "e4m3", None, 152)
    assert s["swap_ab"] == 1
    small = tg.tg_plan_mx(300, 300, 256, 256, 256, 300, "e4m3", None, 152)
    assert small["grid"] == 2 * small["tiles"]
    # lda not a 16-byte multiple: the plain-load producer on 256 x 128 tiles,
    # four more warps; the TMA producer cannot be forced.
    plain = tg.tg_plan_mx(100, 100, 100, 100, 112, 100, "e4m3", None, 152)
    assert plain["producer"] == 2 and plain["block_n"] == 128
    assert plain["threads"] == q["threads"] + 128
    assert tg.tg_plan_mx(100, 100, 100, 112, 112, 100, "e4m3", None, 152)["producer"] == 1
    fp4 = tg.tg_plan_mx(300, 200, 512, 514, 512, 300, "e2m1", None, 152)
    assert fp4["producer"] == 2
    wide = tg.tg_plan_mx(100, 100, 100, 100, 112, 100, "e4m3", {"block_n": 256}, 152)
    assert wide["producer"] == 2 and wide["block_n"] == 256
    with pytest.raises(tg.TgError):
        tg.tg_plan_mx(100, 100, 100, 100, 112, 100, "e4m3", {"producer": 1}, 152)


def test_plan_dynamic_schedule(tg):
    """schedule = 2: CTA-pair tiles, one 2-CTA cluster launched per tile."""
    c4 = si.WORKLOADS["c4_bf16_8192"]
    p = plan(tg, c4, opts={"schedule": 2})
    assert p["cta_pair"] == 1 and p["grid"] == 2 * p["tiles"] == 2048
    assert (p["split_segs"], p["multicast"]) == (1, 1)
    small = plan(tg, si.Workload("s", 500, 500, 2048, "bf16", 1.0, True, 0, "normal"),
                 opts={"schedule": 2, "cta_pair": 2})
    assert small["split_segs"] == 1 and small["grid"] == 2 * small["tiles"]
    with pytest.raises(tg.TgError):      # plain loads: no pair tiles
        plan(tg, si.WORKLOADS["c1_bf16_65x97x73"], opts={"schedule": 2})
    with pytest.raises(tg.TgError):      # TF32 has no pair tiles
        plan(tg, si.WORKLOADS["c2_tf32_256x128x512"], opts={"schedule": 2})


@pytest.mark.parametrize("ops", [
    [(10, 0, 0, None)], [(-1, 0, 0, None)], [("bias_row", 0, 0, None)],
    [("bias_col", 0, 0, FAKE + 2)], [("relu", 0, 0, None)] * 9,
])
def test_epilogue_invalid_ops_rejected_before_cuda(tg, ops):
    st = tg.tg_gemm_epilogue(10, 10, 10, 1.0, FAKE, 10, FAKE, 10, FAKE, 10, "bf16", "f32", ops)
    assert st == tg.TG_ERR_INVALID_VALUE


@pytest.mark.parametrize("args", [
    dict(ssfa=8), dict(ssfb=512 * 7), dict(ssfa=-512), dict(sb=-1024),
    dict(sd=90), dict(batch=-1), dict(ops=[(12, 0, 0, None)]), dict(dtype="bf16"),
    dict(dtype="e2m1", sa=10 * 1024 + 1), dict(sa=8, opts={"producer": 1}),
    dict(dtype="e2m1", sb=10 * 1024 + 16, opts={"producer": 1}),
    dict(opts={"split_k": 2}), dict(out=4), None, dict(sa=8), dict(dtype="e2m1", sb=10 * 1024 + 16),
])
def test_mx_batched_invalid_arguments_rejected_before_cuda(tg, args):
    """Scale strides: 0 or a multiple of 16 at least one entry's atoms;
    operand batch strides even for packed FP4, and of 16-byte multiples when
    the TMA producer is forced; outputs that do not overlap.  The last three
    calls pass validation (and then need a device)."""
    fa = tg.tg_mx_scale_bytes(10, 1024)
    a = dict(sa=10 * 1024, ssfa=fa, sb=10 * 1024, ssfb=fa, sd=10 * 10, batch=3, dtype="e4m3",
             out="f32", ops=[], opts=None)
    a.update(args or {})
    st = tg.tg_gemm_mx_batched(10, 10, 1024, 1.0, FAKE, 1024, a["sa"], FAKE, a["ssfa"], FAKE, 1024,
                               a["sb"], FAKE, a["ssfb"], FAKE, 10, a["sd"], a["batch"], a["dtype"],
                               a["out"], a["ops"], a["opts"])
    if args is None or args in (dict(sa=8), dict(dtype="e2m1", sb=10 * 1024 + 16)):
        assert st != tg.TG_ERR_INVALID_VALUE
    else:
        assert st == tg.TG_ERR_INVALID_VALUE


def test_mx_batched_empty_is_ok_without_cuda(tg):
    assert tg.tg_gemm_mx_batched(0, 10, 64, 1.0, None, 64, 0, None, 0, FAKE, 64, 0, FAKE, 0, None,
                                 1, 0, 4, "e4m3", "f32") == tg.TG_OK
    assert tg.tg_gemm_mx_batched(10, 10, 64, 1.0, FAKE, 64, 0, FAKE, 0, FAKE, 64, 0, FAKE, 0, FAKE,
                                 10, 100, 0, "e4m3", "f32") == tg.TG_OK


def test_plan_stream_k(tg):
    """Stream-K: single-CTA tiles spread over up to every SM (at least 8 K
    blocks each) where the shorter K chain outweighs the fix-up; schedule 1
    or split_k 1 turn it off; schedule 3 forces it."""
    long_k = si.Workload("long_k", 256, 256, 65536, "bf16", 1.0, True, 0, "normal")
    p = plan(tg, long_k)
    assert (p["stream_k"], p["cta_pair"], p["block_n"], p["grid"], p["tiles"]) == (1, 0, 64, 152, 8)
    assert plan(tg, long_k, opts={"max_ctas": 100})["grid"] == 100
    s = plan(tg, long_k, opts={"schedule": 1})
    assert s["stream_k"] == 0
    assert plan(tg, long_k, opts={"split_k": 1})["stream_k"] == 0
    c2 = plan(tg, si.WORKLOADS["c2_tf32_256x128x512"])
    assert (c2["stream_k"], c2["grid"], c2["tiles"]) == (1, 8, 4)        # 2 CTAs per tile
    # Short K chains stay whole: the fix-up would cost more than it saves.
    for name in ("c1_bf16_65x97x73", "c5a_bf16_16384x64x4096", "c5b_bf16_64x16384x4096"):
        assert plan(tg, si.WORKLOADS[name])["stream_k"] == 0, name
    assert plan(tg, si.Workload("k1024", 1024, 1024, 1024, "bf16", 1.0, True, 0, "normal"))[
        "split_segs"] == 1
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"])["stream_k"] == 0          # pair tiles
    one = si.Workload("one", 128, 64, 4096, "bf16", 1.0, True, 0, "normal")
    f = plan(tg, one, opts={"schedule": 3})
    assert (f["stream_k"], f["grid"], f["tiles"]) == (1, 8, 1)            # 64 K blocks / 8
    big = plan(tg, si.WORKLOADS["c3_fp16_4096"], opts={"schedule": 3})
    assert big["stream_k"] == 1 and big["cta_pair"] == 0 and big["grid"] == 152


def test_plan_k_split_pairs_for_mid_shapes(tg):
    """Fewer pair tiles than pairs with a long K loop: the pair split tail
    (K segments on otherwise idle pairs) beats one wave of narrow tiles."""
    for (M, N, K), bn, segs in [((1024, 1024, 8192), 256, 4), ((2048, 512, 16384), 256, 4),
                                ((4096, 128, 8192), 128, 4), ((512, 2048, 4096), 128, 2)]:
        p = plan(tg, si.Workload("mid", M, N, K, "bf16", 1.0, True, 0, "normal"))
        assert (p["cta_pair"], p["block_n"], p["split_segs"]) == (1, bn, segs), (M, N, K)


def test_plan_describe_formats_the_plan(tg):
    w = si.WORKLOADS["c4_bf16_8192"]
    text = tg.tg_plan_describe(w.M, w.N, w.K, w.dtype, *w.strides, 152)
    p = plan(tg, w)
    assert text.startswith("pair 256x256x64 stages=7 producer=tma swap=0 grid=152 tiles=1024 ")
    fields = dict(kv.split("=") for kv in text.split()[2:])
    assert int(fields["tiles"]) == p["tiles"] and int(fields["raster"]) == p["raster_group"]
    assert fields["split"] == f"{p['split_tiles']}x{p['split_segs']}"
    assert int(fields["smem"]) == p["smem_bytes"] and int(fields["tmem"]) == p["tmem_cols"]
    c1 = si.WORKLOADS["c1_bf16_65x97x73"]
    assert tg.tg_plan_describe(c1.M, c1.N, c1.K, c1.dtype, *c1.strides, 152).startswith(
        "single 128x64x64 stages=8 producer=plain")
    assert tg.tg_plan_describe(0, 5, 5, "bf16", 5, 5, 1, 152) == "empty"


def test_plan_describe_errors(tg):
    import ctypes

    lib = tg.load()
    small = ctypes.create_string_buffer(16)
    # Too small: truncated, NUL-terminated, and reported.
    assert lib.tg_plan_describe(8192, 8192, 8192, 0, 8192, 8192, 8192, 152, small, 16) == \
        tg.TG_ERR_INVALID_VALUE
    assert small.value == b"pair 256x256x64"
    assert lib.tg_plan_describe(8, 8, 8, 0, 8, 8, 8, 152, None, 16) == tg.TG_ERR_INVALID_VALUE
    assert lib.tg_plan_describe(8, 8, 8, 0, 7, 8, 8, 152, small, 16) == tg.TG_ERR_INVALID_VALUE
    with pytest.raises(tg.TgError):
        tg.tg_plan_describe(8, 8, 8, "bf16", 8, 8, 8, 152, size=8)


def test_plan_ticket_schedule(tg):
    """Tickets from 6 waves of CTA-pair tiles up (one pair per cluster);
    fewer waves run static, both with the exchange split of a last wave at
    most half full."""
    c3 = plan(tg, si.WORKLOADS["c3_fp16_4096"])          # 256 tiles on 76 pairs: 3.4 waves
    assert (c3["cta_pair"], c3["multicast"], c3["schedule"]) == (1, 1, 1)
    assert (c3["split_tiles"], c3["split_segs"]) == (28, 2)
    assert plan(tg, si.WORKLOADS["c3_fp16_4096"], opts={"schedule": 4})["schedule"] == 4
    c4 = plan(tg, si.WORKLOADS["c4_bf16_8192"])          # 13.5 waves
    assert (c4["schedule"], c4["split_tiles"], c4["split_segs"]) == (4, 36, 2)
    six = plan(tg, si.Workload("s", 256 * 19, 256 * 24, 4096, "bf16", 1.0, True, 0, "normal"))
    assert (six["tiles"], six["schedule"]) == (456, 4)   # exactly 6 waves of 76 pairs
    five = plan(tg, si.Workload("s", 256 * 19, 256 * 20, 4096, "bf16", 1.0, True, 0, "normal"))
    assert (five["tiles"], five["schedule"]) == (380, 1)
    # Multicast clusters and fewer tiles than pairs stay static.
    assert plan(tg, si.WORKLOADS["c5c_bf16_8191x4097x1000"])["schedule"] == 1
    few = plan(tg, si.Workload("f", 1000, 1000, 4096, "bf16", 1.0, True, 0, "normal"))
    assert few["cta_pair"] == 1 and few["schedule"] == 1
    # Forced where it cannot run (fewer tiles than pairs): refused.
    with pytest.raises(tg.TgError):
        plan(tg, si.Workload("f", 1000, 1000, 4096, "bf16", 1.0, True, 0, "normal"),
             opts={"schedule": 4})
    # Single-CTA plans report static or stream-K.
    assert plan(tg, si.WORKLOADS["c5a_bf16_16384x64x4096"])["schedule"] == 1
    assert plan(tg, si.WORKLOADS["c2_tf32_256x128x512"])["schedule"] == 3


def test_plan_k_snake(tg):
    """16-bit CTA-pair tiles under tickets alternate their K order by wave;
    the static schedule, the 8-bit kinds, two-pair clusters and single-CTA
    tiles keep ascending K."""
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"])["k_snake"] == 1
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"schedule": 1})["k_snake"] == 0
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"split_k": 1})["k_snake"] == 0
    assert plan(tg, si.WORKLOADS["c4_bf16_8192"], opts={"schedule": 2})["k_snake"] == 0
    assert plan(tg, si.WORKLOADS["c3_fp16_4096"], opts={"schedule": 4})["k_snake"] == 1
    for name in ("c3_fp16_4096", "f8_e4m3_8192", "c5c_bf16_8191x4097x1000",
                 "c5a_bf16_16384x64x4096", "c1_bf16_65x97x73"):
        assert plan(tg, si.WORKLOADS[name])["k_snake"] == 0, name
    w = si.WORKLOADS["c4_bf16_8192"]
    assert " k_snake=1 " in tg.tg_plan_describe(w.M, w.N, w.K, w.dtype, *w.strides, 152)


def test_plan_k_rotate(tg):
    """One wave of single-CTA whole tiles walks each tile's K blocks from its
    own offset, where the operand the tiles share fits in L2."""
    for name in ("c5a_bf16_16384x64x4096", "c5b_bf16_64x16384x4096"):
        p = plan(tg, si.WORKLOADS[name])
        assert (p["cta_pair"], p["k_rotate"]) == (0, 1)
        assert plan(tg, si.WORKLOADS[name], opts={"schedule": 1})["k_rotate"] == 0
        assert plan(tg, si.WORKLOADS[name], opts={"schedule": 3})["k_rotate"] == 0
    for name in ("c4_bf16_8192", "c3_fp16_4096", "c2_tf32_256x128x512", "c1_bf16_65x97x73"):
        assert plan(tg, si.WORKLOADS[name])["k_rotate"] == 0    # (c1: a 2-block K loop)
    # More tiles than CTAs (several waves): no rotation.
    many = plan(tg, si.Workload("m", 4096, 4096, 4096, "bf16", 1.0, True, 0, "normal"),
                opts={"cta_pair": 1})
    assert many["tiles"] > many["grid"] and many["k_rotate"] == 0
    # One wave whose shared A-role operand is large (two N blocks of a tall A): no rotation.
    w = si.Workload("t", 8192, 512, 8192, "bf16", 1.0, True, 0, "normal")
    tall = plan(tg, w, opts={"cta_pair": 1, "block_n": 256, "split_k": 1})
    assert tall["tiles"] <= tall["grid"] and tall["stream_k"] == 0 and tall["k_rotate"] == 0
    # The same wave with a small A-role operand rotates.
    short = plan(tg, si.with_shape(w, M=1024, K=2048, lda=2048, ldb=2048),
                 opts={"cta_pair": 1, "block_n": 128, "split_k": 1})
    assert short["tiles"] <= short["grid"] and short["k_rotate"] == 1
