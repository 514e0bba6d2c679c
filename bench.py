#!/usr/bin/env python3
"""Benchmark: BF16 GEMM + ReLU at M = N = K = 8192 through the tg_gemm C ABI.

One step is one call of the whole path (plan, TMA descriptors, the persistent
tcgen05 kernel with its fused alpha/ReLU epilogue) over the 8192^3 workload:
A, B BF16 (seeded standard normal), D FP32 column-major, alpha = 1.  Inputs
stay resident in HBM; A + B (268 MB) and D (268 MB) are each larger than the
129 MB L2, so no flush is needed between steps.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the
only other arm), on a bounded sample of the same workload.

Workloads whose inputs are smaller than twice the L2 (``--workload``, and the
other configurations the default run also times, under ``other_workloads``)
cycle through several device copies of their inputs and outputs between
launches, so that no launch finds its inputs in L2; where that would take
more than 16 copies (the small latency-bound shapes) the L2 is flushed by a
256 MB write before each launch instead, with events around every launch.

The library is single-GPU: some of its kernels load operand tiles with
cluster-multicast TMA, which is used only by calls that run on one GPU.  The
GPU arm therefore refuses to run with more than one GPU (``--gpus`` other
than 1, or a ``WORLD_SIZE`` above 1) and exits non-zero.  The reference arm
never touches a GPU; under a multi-rank launch rank 0 runs it and the other
ranks exit without work.
"""

from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

WORKLOAD = "c4_bf16_8192"
METRIC = "bf16 GEMM+ReLU TFLOP/s at 8192³; % of GB300 dense BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
L2_BYTES = 129e6
FLUSH_BYTES = 256 << 20
MAX_COPIES = 16
# The other configurations of the library's workload table, timed after the
# headline in the default run (20 launches each after 5 warm-up).
OTHER_WORKLOADS = ["c1_bf16_65x97x73", "c2_tf32_256x128x512", "c3_fp16_4096",
                   "c5a_bf16_16384x64x4096", "c5b_bf16_64x16384x4096", "c5c_bf16_8191x4097x1000"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs to use; the GPU arm runs on exactly one")
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="tg", choices=["tg", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(si.WORKLOADS),
                    help="problem to time (default: the 8192^3 BF16 + ReLU headline)")
    ap.add_argument("--out", default="f32", choices=["f32", "bf16", "fp16"],
                    help="output type of D (bf16/fp16 go through tg_gemm_batched)")
    ap.add_argument("--batch", type=int, default=1,
                    help="batch entries of the workload per step (tg_gemm_batched)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip timing the other configurations in the default run")
    ap.add_argument("--cpu-baseline", action="store_true",
                    help="time the oracle also for a non-default workload")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def single_gpu_refusal(args, world: int) -> str | None:
    """Why the GPU arm must not run with these arguments, or None.  Both
    --gpus and WORLD_SIZE must say one GPU: the library's multicast loads are
    for single-GPU calls only, so there is no replica mode."""
    if args.gpus != 1 or world != 1:
        return (f"single-GPU library: replicas not run (--gpus {args.gpus}, WORLD_SIZE {world}); "
                f"the GPU arm runs on exactly one GPU")
    return None


def workload_config(w: si.Workload, world: int, out: str = "f32", batch: int = 1) -> dict:
    lda, ldb, ldc = w.strides
    scales = ""
    if w.block_scaled and w.dtype == "nvf4":
        lo, hi = si.bench_scales(w.dtype)
        scales = (f", one unsigned-E4M3 scale per 16 K (seeded codes 0x{lo:02X}..0x{hi:02X}: "
                  f"0.25..4)")
    elif w.block_scaled:
        lo, hi = si.bench_scales(w.dtype)
        scales = (f", one 8-bit exponent scale per 32 K (seeded codes {lo}..{hi}: "
                  f"2^{lo - 127}..2^{hi - 127})")
    dist = ("N(0,1)" + (f"x{w.scale}" if w.scale != 1.0 else "") if w.dist == "normal"
            else f"U[{w.lo},{w.hi})")
    cfg = {
        "workload": f"{w.name}: M={w.M} N={w.N} K={w.K} {w.dtype.upper()} operands (seeded "
                    f"{dist}){scales}, alpha={w.alpha}, {'ReLU' if w.relu else 'no'} epilogue, FP32 "
                    f"accumulate, D {out.upper()} column-major"
                    + (f", batch of {batch} (entries share one seeded draw)" if batch > 1 else ""),
        "M": w.M, "N": w.N, "K": w.K, "lda": lda, "ldb": ldb, "ldc": ldc,
        "parallelism": "single GPU",
    }
    if batch > 1:
        cfg["batch"] = batch
    if out != "f32":
        cfg["out"] = out
    e = si.element_bytes(w.dtype)
    ws = batch * ((w.M * w.K + w.K * w.N) * e + w.M * w.N * (4 if out == "f32" else 2))
    ins = batch * (w.M * w.K + w.K * w.N) * e
    n = input_copies(ins)
    cfg["l2"] = (f"inputs {ins / 1e6:.3g} MB, working set {ws / 1e6:.3g} MB vs 129 MB L2; " +
                 ("inputs larger than twice the L2, no flush" if n == 1 else
                  f"launches cycle through {n} copies of inputs and output "
                  f"({n * ins / 1e6:.0f} MB of inputs)" if n else
                  "L2 flushed by a 256 MB write before each launch (events around each launch)"))
    return cfg


def input_copies(in_bytes: float) -> int:
    """Device copies of a workload's inputs (and output) that the timed
    launches cycle through: 1 when the inputs alone are at least twice the
    L2; else enough copies to reach that; 0 (flush the L2 before each launch
    instead) when that would take more than MAX_COPIES."""
    if in_bytes >= 2 * L2_BYTES:
        return 1
    n = math.ceil(2 * L2_BYTES / max(in_bytes, 1.0))
    return n if n <= MAX_COPIES else 0


def time_launches(torch, launch, n_sets: int, steps: int, stream, flush=None):
    """Average milliseconds per launch of `launch(i)` over `steps` launches.
    n_sets >= 1: back-to-back launches between two events on `stream`, launch
    i on input set i % n_sets.  n_sets == 0: `flush` (a buffer larger than
    the L2) is overwritten before every launch and events surround each
    launch alone; the average of those."""
    if n_sets:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(steps):
            launch(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            launch(i)
            ends[i].record(stream)
    torch.cuda.synchronize()
    return statistics.fmean(s.elapsed_time(e) for s, e in zip(starts, ends))


def roofline(w: si.Workload, ms: float, peaks: dict, sustained: bool, out: str = "f32",
             nbat: int = 1) -> dict:
    """The workload's bound (tensor or HBM, by its arithmetic intensity
    against the peaks' ridge point) and the fraction of that peak one launch
    of `ms` milliseconds reaches.  TF32, the 8-bit and the 4-bit floats take
    the BF16 peak times the nominal ratio to BF16 (1.1, 4.5 and 13.5 over
    2.25 PFLOP/s)."""
    flops = w.flops * nbat
    alg_bytes = nbat * ((w.M * w.K + w.K * w.N) * si.element_bytes(w.dtype) +
                        w.M * w.N * (4 if out == "f32" else 2))
    if w.block_scaled:   # one scale byte per block of K
        alg_bytes += nbat * (w.M + w.N) * (-(-w.K // si.scale_block(w.dtype)))
    ratio = {"tf32": 1.1 / 2.25, "e4m3": 4.5 / 2.25, "e5m2": 4.5 / 2.25,
             "e2m1": 13.5 / 2.25, "nvf4": 13.5 / 2.25}.get(w.dtype, 1.0)
    note = {"tf32": " x 1.1/2.25 (TF32)", "e4m3": " x 4.5/2.25 (FP8)",
            "e5m2": " x 4.5/2.25 (FP8)", "e2m1": " x 13.5/2.25 (FP4)",
            "nvf4": " x 13.5/2.25 (FP4)"}.get(w.dtype, "")
    sustained = sustained and "bf16_tflops_sustained" in peaks
    tpeak = ratio * float(peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    tensor = flops / alg_bytes >= tpeak * 1e12 / (hbm * 1e9)
    if tensor:
        achieved, peak, unit = flops / (ms * 1e-3) / 1e12, tpeak, "TFLOP/s"
        src = ("bf16_tflops_sustained" if sustained else "bf16_tflops (burst)") + note
    else:
        achieved, peak, unit = alg_bytes / (ms * 1e-3) / 1e9, hbm, "GB/s"
        src = "hbm_gbs"
    return {"bound": "tensor" if tensor else "hbm", "achieved": achieved, "peak": peak,
            "unit": unit, "frac": achieved / peak, "peak_field": src,
            "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": alg_bytes}


# ------------------------------------------------------------------ oracle timing

def oracle_sample_time(w: si.Workload, A, B, rows: int, cols: int, threads: int = 0) -> float:
    """Wall time of the oracle on the leading block D[0:rows, 0:cols] of the
    workload (full K): the same arithmetic those entries get in the full
    problem, since D[i, j] reads only row i of A and column j of B."""
    import oracle

    lda, ldb, _ = w.strides
    As = np.ascontiguousarray(A[:rows])
    Bs = np.ascontiguousarray(B[:cols])
    if w.block_scaled:
        SA, SB = si.make_mx_scales(si.with_shape(w, M=rows, N=cols))
        kb = SA.shape[1]
        t0 = time.perf_counter()
        oracle.gemm_mx(rows, cols, w.K, w.alpha, As, lda, SA, kb, Bs, ldb, SB, kb, w.dtype, w.relu,
                       threads=threads)
        return time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.gemm(rows, cols, w.K, w.alpha, As, lda, Bs, ldb, w.dtype, w.relu, threads=threads)
    return time.perf_counter() - t0


def calibrate_block(w, A, B, target_s: float) -> int:
    """Square sample size whose oracle time is about target_s (timed first on
    a 512 x 512 sample: smaller ones overstate the cost per entry, their
    columns leaving host threads idle)."""
    c = int(min(512, w.M, w.N))
    t = oracle_sample_time(w, A, B, c, c)
    per_entry = max(t / (float(c) * c), 1e-9)
    s = int((target_s / per_entry) ** 0.5) // 64 * 64
    return int(max(64, min(s, w.M, w.N)))


def cpu_baseline(w: si.Workload, A, B, target_s: float = 15.0) -> dict:
    import oracle

    s = calibrate_block(w, A, B, target_s)
    t = oracle_sample_time(w, A, B, s, s)
    flops = 2.0 * s * s * w.K
    return {
        "value": flops / t / 1e12, "unit": UNIT, "cores": oracle.host_threads(), "kind": "oracle",
        "sample": f"D[0:{s}, 0:{s}] of the {w.M}x{w.N}x{w.K} workload (full K), {t:.1f} s wall "
                  f"on the host cores, double-precision C triple loop",
    }


def metric_name(w: si.Workload, nbat: int = 1, out: str = "f32") -> str:
    """The headline metric for the benchmark workload; for any other workload
    the same quantity (TFLOP/s) named by its type, epilogue and shape."""
    if w.name == WORKLOAD and nbat == 1 and out == "f32":
        return METRIC
    blocks = f"block-scaled ({si.scale_block(w.dtype)}-element blocks) " if w.block_scaled else ""
    return (f"{blocks}"
            f"{w.dtype} GEMM{'+ReLU' if w.relu else ''} TFLOP/s at {w.M}x{w.N}x{w.K}"
            + (f" x{nbat}" if nbat > 1 else "") + (f", {out} out" if out != "f32" else ""))


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, timed on the host cores
    on a bounded square sample D[0:s, 0:s] (full K) of the chosen workload."""
    if rank != 0:
        return 0
    if args.batch != 1 or args.out != "f32":
        raise SystemExit("--impl reference times the unbatched product with FP32 output")
    w = si.WORKLOADS[args.workload]
    A, B = si.make_operands(w)
    import oracle

    # Size each step so that (warmup + steps) steps end within ~2.5 minutes.
    per_step_target = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    blk = calibrate_block(w, A, B, per_step_target)
    for _ in range(args.warmup):
        oracle_sample_time(w, A, B, blk, blk)
    times = [oracle_sample_time(w, A, B, blk, blk) for _ in range(args.steps)]
    total = sum(times)
    flops = 2.0 * blk * blk * w.K
    value = flops * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": metric_name(w), "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.host_threads(),
                         "kind": "oracle",
                         "sample": f"each step: D[0:{blk}, 0:{blk}] of the {w.M}x{w.N}x{w.K} "
                                   f"workload (full K), double-precision C triple loop on the "
                                   f"host cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    # power.draw is averaged over about a second, longer than the timed region;
    # the instantaneous reading is taken too where this nvidia-smi knows it.
    INSTANT = "power.draw.instant"

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        self.instant = False

    def _knows_instant(self) -> bool:
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.index),
                                f"--query-gpu={self.INSTANT}", "--format=csv,noheader,nounits"],
                               capture_output=True, text=True, timeout=20)
        except (OSError, subprocess.SubprocessError):
            return False
        try:
            float(r.stdout.strip().splitlines()[0])
        except (ValueError, IndexError):
            return False
        return r.returncode == 0

    def start(self):
        self.instant = self._knows_instant()
        query = self.QUERY + ("," + self.INSTANT if self.instant else "")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={query}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = list(csv.reader(io.StringIO(out)))
        samples = []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + r[0].strip().split(".")[1]) if "." in r[0] else 0.0
                samples.append((ts + frac, [x.strip() for x in r]))
            except (ValueError, IndexError):
                continue
        inside = [s for t, s in samples if self.t0 - 0.05 <= t <= self.t1 + 0.05]
        use = inside or [s for _, s in samples]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(s[2]) for s in use if s[2].replace(".", "").isdigit()]
        smax = [float(s[3]) for s in use if s[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in use for i in range(4) if s[6 + i] == "Active"})
        col = 10 if self.instant else 4
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(inside),
                "power_w_max": max((float(s[col]) for s in use
                                    if len(s) > col and s[col].replace(".", "").isdigit()),
                                   default=None),
                "power_field": self.INSTANT if self.instant else "power.draw"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(kernel_hash: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the kernel as it is now (same source hash); else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(WORKLOAD)
    if not e or e.get("source_hash") != kernel_hash:
        return None
    return e.get("dram_bytes_per_launch")


def run_gpu(args):
    import torch

    import dense_gemm_epilogue_gb300 as tg

    torch.cuda.set_device(0)
    tg.build()
    tg.load()
    w = si.WORKLOADS[args.workload]
    out, nbat = args.out, max(1, args.batch)
    batched = nbat > 1 or out != "f32"
    lda, ldb, ldc = w.strides
    A, B = si.make_operands(w)
    view = {"tf32": np.float32, "e4m3": np.uint8, "e5m2": np.uint8,
            "e2m1": np.uint8, "nvf4": np.uint8}.get(w.dtype, np.int16)
    hA = torch.from_numpy(np.tile(A.reshape(-1), nbat).view(view)).pin_memory()
    hB = torch.from_numpy(np.tile(B.reshape(-1), nbat).view(view)).pin_memory()
    dA = hA.cuda()
    dB = hB.cuda()
    odt = torch.float32 if out == "f32" else torch.int16
    dD = torch.empty((nbat * w.N, ldc), dtype=odt, device="cuda")
    hD = torch.empty((nbat * w.N, ldc), dtype=odt).pin_memory()
    sa, sb, sd = w.M * lda, w.N * ldb, w.N * ldc   # elements (unused for block-scaled FP4)
    stream = torch.cuda.Stream()
    mx = w.block_scaled
    if mx:
        if batched:
            raise SystemExit("block-scaled workloads run unbatched with FP32 output")
        # Scale atoms, packed on the device by the library from the seeded
        # row-major scales; they are inputs like A and B (uploaded in e2e).
        SA, SB = si.make_mx_scales(w)
        dSA = torch.empty(tg.tg_bs_scale_bytes(w.M, w.K, w.dtype), dtype=torch.uint8,
                          device="cuda")
        dSB = torch.empty(tg.tg_bs_scale_bytes(w.N, w.K, w.dtype), dtype=torch.uint8,
                          device="cuda")
        tg.check(tg.tg_bs_pack_scales(w.M, w.K, w.dtype, torch.from_numpy(SA).cuda(), SA.shape[1],
                                      dSA), "tg_bs_pack_scales")
        tg.check(tg.tg_bs_pack_scales(w.N, w.K, w.dtype, torch.from_numpy(SB).cuda(), SB.shape[1],
                                      dSB), "tg_bs_pack_scales")
        torch.cuda.synchronize()
        hSA, hSB = dSA.cpu().pin_memory(), dSB.cpu().pin_memory()
        plan = tg.tg_plan_mx(w.M, w.N, w.K, lda, ldb, ldc, w.dtype)
    else:
        plan = tg.tg_plan(w.M, w.N, w.K, dA, lda, dB, ldb, None, ldc, w.dtype)
    scale_inputs = {}
    # Input sets the timed launches cycle through (see input_copies).
    in_bytes = hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
    n_sets = input_copies(in_bytes)
    sets = [(dA, dB, dD)]
    for _ in range(1, n_sets):
        sets.append((dA.clone(), dB.clone(), torch.empty_like(dD)))
        if mx:
            scale_inputs[sets[-1][0].data_ptr()] = (dSA.clone(), dSB.clone())
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda") if n_sets == 0 else None

    def call(a_, b_, d_, st_):
        if mx:
            sfa, sfb = scale_inputs.get(a_.data_ptr(), (dSA, dSB))
            return tg.tg_gemm_mx(w.M, w.N, w.K, w.alpha, a_, lda, sfa, b_, ldb, sfb, d_, ldc,
                                 w.dtype, "f32", w.relu, None, st_)
        if batched:
            return tg.tg_gemm_batched(w.M, w.N, w.K, w.alpha, a_, lda, sa, b_, ldb, sb, d_, ldc, sd,
                                      nbat, w.dtype, out, w.relu, None, st_)
        return tg.tg_gemm(w.M, w.N, w.K, w.alpha, a_, lda, b_, ldb, d_, ldc, w.dtype, w.relu, st_)

    def step(i=0):
        a_, b_, d_ = sets[i % len(sets)]
        st = call(a_, b_, d_, stream)
        if st != tg.TG_OK:
            raise tg.TgError(st, "tg_gemm")

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()

    # The timed region: exactly `steps` back-to-back calls, one kernel launch
    # each, bracketed by two events on the launching stream.  Nothing else is
    # recorded between the launches, so each kernel's prologue overlaps the
    # previous one's tail (programmatic dependent launch) as in any sequence
    # of calls; the kernel's average launch duration is region / steps.
    # (Inputs smaller than the L2: see input_copies and time_launches.)
    sampler = ClockSampler(0)
    sampler.start()
    sampler.mark("t0")
    region_ms = args.steps * time_launches(torch, step, n_sets, args.steps, stream, flush)
    sampler.mark("t1")
    st, where = tg.tg_check_device_status(stream)
    if st != tg.TG_OK:
        raise tg.TgError(st, f"device status (wait site {where})")
    clocks = sampler.stop()

    # A separate, untimed pass with events around every launch gives the
    # spread of single launches (an event between two launches stops the
    # overlap above, so these read a little slower than the timed region).
    n_each = min(args.steps, 50)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_each)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_each)]
    for i in range(n_each):
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # End to end through the public API: every step copies its inputs A, B
    # from pinned host memory, runs the call and reads D back to pinned host
    # memory.  Steps are pipelined over two device buffer sets on three
    # streams (H2D, compute, D2H), so step i+1's upload overlaps step i's
    # download; the time is from the first upload to the last download.
    e2e_steps = max(2, args.e2e_steps)
    bufs = [(dA, dB, dD)]
    bufs.append((torch.empty_like(dA), torch.empty_like(dB), torch.empty_like(dD)))
    if mx:
        scale_bufs = [(dSA, dSB), (torch.empty_like(dSA), torch.empty_like(dSB))]
        for (a_, _, _), sc in zip(bufs, scale_bufs):
            scale_inputs[a_.data_ptr()] = sc
    hDs = [hD, torch.empty_like(hD).pin_memory()]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_gemm = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        a_, b_, d_ = bufs[b]
        if i >= 2:
            s_in.wait_event(ev_gemm[b])          # step i-2 has finished reading A, B
        with torch.cuda.stream(s_in):
            a_.copy_(hA, non_blocking=True)
            b_.copy_(hB, non_blocking=True)
            if mx:
                sfa_, sfb_ = scale_bufs[b]
                sfa_.copy_(hSA, non_blocking=True)
                sfb_.copy_(hSB, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])         # step i-2's D has been read back
        st_ = call(a_, b_, d_, stream)
        if st_ != tg.TG_OK:
            raise tg.TgError(st_, "tg_gemm")
        ev_gemm[b].record(stream)
        s_out.wait_event(ev_gemm[b])
        with torch.cuda.stream(s_out):
            hDs[b].copy_(d_, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.perf_counter()
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_wall = time.perf_counter() - t_wall0
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    step_ms = region_ms / args.steps

    flops = w.flops * nbat
    value = flops / (step_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    launch_avg_ms = step_ms  # one kernel launch per step
    # Back-to-back launches for more than ~50 ms run in the power-capped
    # regime the sustained peak was measured in; a short burst compares
    # with the burst peak.
    sustained = region_ms > 50.0 and n_sets != 0 and "bf16_tflops_sustained" in peaks
    rf = roofline(w, launch_avg_ms, peaks, sustained, out, nbat)
    tensor_bound = rf["bound"] == "tensor"
    qs = sorted(launch_ms)
    each = {"launches": len(launch_ms), "avg_ms": statistics.fmean(launch_ms),
            "p10_p50_p90_ms": [qs[len(qs) // 10], qs[len(qs) // 2], qs[(9 * len(qs)) // 10]],
            "how": "separate untimed pass after the timed region, events around every launch"}
    if tensor_bound and sustained:
        each["frac_of_burst_peak"] = roofline(w, each["avg_ms"], peaks, False, out, nbat)["frac"]
    dt = w.dtype
    kname = ("tg_gemm_mx_kernel" if mx else
             "tg_gemm_pair_kernel" if plan.get("cta_pair") else "tg_gemm_kernel") + \
        f"<{dt.upper()}, {plan['block_m']}x{plan['block_n']}, " + \
        f"{'TMA' if plan['producer'] == 1 else 'plain loads'}>"
    traffic = load_traffic(tg.source_hash()) if args.workload == WORKLOAD and not batched else None
    default_run = args.workload == WORKLOAD and not batched
    line = {
        "metric": metric_name(w, nbat, out),
        "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dt, "data": "synthetic", "config": workload_config(w, 1, out, nbat),
        "roofline": {"bound": rf["bound"], "achieved": rf["achieved"],
                     "peak": rf["peak"], "unit": rf["unit"],
                     "frac": rf["frac"], "traffic": traffic,
                     "peak_source": rf["peak_field"] + f" of {peak_src}" +
                                    (f" (the timed region ran {region_ms:.0f} ms of back-to-back "
                                     f"launches)" if tensor_bound and sustained else ""),
                     "kernel": kname,
                     "kernel_ms_avg": launch_avg_ms,
                     "kernel_ms_how": ("timed region / steps (one launch per step, events on "
                                       "the launching stream around the region)" if n_sets else
                                       "average of events around each launch, each after a "
                                       "256 MB write that flushes the L2"),
                     "per_launch_events": each,
                     "algorithmic_flops_per_launch": rf["algorithmic_flops_per_launch"],
                     "algorithmic_bytes_per_launch": rf["algorithmic_bytes_per_launch"]},
        "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(hA.numel() * hA.element_size() +
                                          hB.numel() * hB.element_size() +
                                          (hSA.numel() + hSB.numel() if mx else 0)),
                "d2h_bytes_per_step": int(hD.numel() * hD.element_size()),
                "steps": e2e_steps, "wall_s": e2e_wall,
                "pipelining": "2 buffer sets; H2D, compute and D2H on separate streams"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "plan": plan,
        "library_source_hash": tg.source_hash(),
    }
    if default_run and not args.no_others:
        del sets, bufs, hDs
        line["other_workloads"] = time_others(torch, tg, peaks, peak_src)
    if not args.no_cpu_baseline and (default_run or args.cpu_baseline):
        line["cpu_baseline"] = cpu_baseline(w, A, B)
    print(json.dumps(line), flush=True)
    return 0


def time_others(torch, tg, peaks: dict, peak_src: str, steps: int = 20, warmup: int = 5) -> dict:
    """The other configurations through tg_gemm, each on its seeded inputs
    (the same recipe as the headline's), `steps` launches after `warmup`,
    timed as the headline (input copies or an L2 flush per input_copies),
    against the burst peaks; clocks sampled over the whole pass."""
    stream = torch.cuda.Stream()
    sampler = ClockSampler(0)
    sampler.start()
    sampler.mark("t0")
    rows = []
    view = {"tf32": np.float32}
    for name in OTHER_WORKLOADS:
        w = si.WORKLOADS[name]
        lda, ldb, ldc = w.strides
        A, B = si.make_operands(w)
        dA = torch.from_numpy(A.reshape(-1).view(view.get(w.dtype, np.int16))).cuda()
        dB = torch.from_numpy(B.reshape(-1).view(view.get(w.dtype, np.int16))).cuda()
        n_sets = input_copies(A.nbytes + B.nbytes)
        sets = [(dA, dB, torch.empty((w.N, ldc), dtype=torch.float32, device="cuda"))]
        for _ in range(1, n_sets):
            sets.append((dA.clone(), dB.clone(), torch.empty_like(sets[0][2])))
        flush = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda") if n_sets == 0
                 else None)

        def launch(i, sets=sets, w=w, lda=lda, ldb=ldb, ldc=ldc):
            a_, b_, d_ = sets[i % len(sets)]
            st = tg.tg_gemm(w.M, w.N, w.K, w.alpha, a_, lda, b_, ldb, d_, ldc, w.dtype, w.relu,
                            stream)
            if st != tg.TG_OK:
                raise tg.TgError(st, "tg_gemm")

        with torch.cuda.stream(stream):
            for i in range(warmup):
                launch(i)
        ms = time_launches(torch, launch, n_sets, steps, stream, flush)
        st, where = tg.tg_check_device_status(stream)
        if st != tg.TG_OK:
            raise tg.TgError(st, f"device status (wait site {where})")
        rf = roofline(w, ms, peaks, False)
        rows.append({
            "workload": name, "ms_per_launch": ms,
            "value": w.flops / (ms * 1e-3) / 1e12, "unit": UNIT,
            "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac")},
            "peak_source": rf["peak_field"] + f" of {peak_src}",
            "l2": workload_config(w, 1)["l2"],
            "plan": tg.tg_plan_describe(w.M, w.N, w.K, w.dtype, lda, ldb, ldc),
        })
        del sets, flush, dA, dB
        torch.cuda.synchronize()
    sampler.mark("t1")
    return {"launches_each": steps, "warmup_each": warmup,
            "how": "one configuration after another, after the headline's timed region",
            "results": rows, "clocks": sampler.stop()}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    why = single_gpu_refusal(args, world)
    if why:
        print(why, file=sys.stderr, flush=True)
        return 2
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
