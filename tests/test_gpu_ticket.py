"""The ticket schedule of the CTA-pair kernel (each pair's first tile is
static, later units are claimed in order from a counter in the stream's
workspace) and the two-segment exchange that finishes a partial last wave,
against the oracle element by element.

Small problems get several waves of pair tiles by capping the grid
(tg_options.max_ctas).  Each case runs three times in a row on one stream:
the results must be bitwise identical (the counter and the exchange flags
are back at zero after every launch, and the exchange adds the two K
segments' partial sums in a fixed order).
"""

from __future__ import annotations

import pytest

import seeded_inputs as si
from gemm_harness import check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()
    return tg


def find_cap(tg, w, want_segs, extra=None):
    """A grid cap (CTAs) under which the planner runs `w` with tickets and
    `want_segs` K segments for the last wave."""
    lda, ldb, ldc = w.strides
    for cap in range(4, 153, 2):
        opts = {"max_ctas": cap, "cta_pair": 2, "schedule": 4, **(extra or {})}
        try:
            p = tg.tg_plan(w.M, w.N, w.K, None, lda, None, ldb, None, ldc, w.dtype, opts)
        except tg.TgError:
            continue
        if p["schedule"] == 4 and p["split_segs"] == want_segs and p["grid"] // 2 >= 2:
            return opts, p
    raise AssertionError(f"no grid cap gives tickets with {want_segs} segments for {w.name}")


CASES = [
    # (workload, K segments of the last wave, extra options); row strides are
    # 16-byte multiples (pair tiles load by TMA), K ragged against the stage.
    (si.Workload("tk_exchange", 1000, 1100, 1100, "bf16", 1.5, True, 81, "uniform", lda=1104,
                 ldb=1104, ldc=1004), 2, None),
    (si.Workload("tk_whole", 1000, 1100, 1100, "bf16", 1.0, True, 82, "normal", lda=1104,
                 ldb=1104), 1, None),
    (si.Workload("tk_bn128", 777, 1500, 1300, "fp16", -0.75, True, 83, "normal", scale=0.5,
                 lda=1304, ldb=1304, ldc=780), 2, {"block_n": 128}),
    (si.Workload("tk_e4m3", 900, 1300, 2100, "e4m3", 0.25, False, 84, "normal", lda=2112,
                 ldb=2112), 2, None),
    (si.Workload("tk_swap", 100, 3000, 1500, "bf16", 1.0, True, 85, "uniform", lda=1504,
                 ldb=1504, ldc=104), 2, None),
]


@pytest.mark.parametrize("w,segs,extra", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_ticket_schedule_parity(tg, w, segs, extra):
    opts, p = find_cap(tg, w, segs, extra)
    assert p["cta_pair"] == 1 and p["multicast"] == 1
    # 16-bit kinds: tiles of odd waves walk K downwards (k_snake).
    assert p["k_snake"] == (1 if w.dtype in ("bf16", "fp16") else 0)
    assert p["tiles"] >= p["grid"]  # at least one tile past the first wave
    check_full(w, opts=opts, repeats=3)


def test_ticket_counter_resets_between_shapes(tg):
    """Different ticket shapes back to back on one stream: each launch starts
    from a zero counter left by the one before."""
    ws = [c[0] for c in CASES[:3]]
    for _ in range(2):
        for w, segs, extra in CASES[:3]:
            opts, _ = find_cap(tg, w, segs, extra)
            check_full(w, opts=opts)


def test_ticket_forced_matches_static(tg):
    """schedule = 4 on a full-size wave count, against the oracle; the static
    schedule on the same problem gives results within the same tolerance."""
    w = si.Workload("tk_forced", 2560, 2304, 1536, "bf16", 1.0, True, 86, "normal")
    check_full(w, opts={"schedule": 4})
    check_full(w, opts={"schedule": 1})


def test_static_exchange_split_parity(tg):
    """The static schedule with the two-segment exchange of a last wave at
    most half full (the planner's choice for a few waves of pair tiles)."""
    w = si.Workload("st_exchange", 1000, 1100, 1100, "bf16", 1.25, True, 87, "normal", lda=1104,
                    ldb=1104, ldc=1001)
    lda, ldb, ldc = w.strides
    for cap in range(4, 153, 2):
        opts = {"max_ctas": cap, "cta_pair": 2, "schedule": 1}
        p = tg.tg_plan(w.M, w.N, w.K, None, lda, None, ldb, None, ldc, w.dtype, opts)
        if p["split_segs"] == 2 and p["tiles"] >= p["grid"] // 2:
            break
    else:
        raise AssertionError("no grid cap gives a static exchange split")
    assert p["schedule"] == 1
    check_full(w, opts=opts, repeats=3)
