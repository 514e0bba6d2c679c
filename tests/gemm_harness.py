"""Shared test plumbing: run tg_gemm through the C ABI on numpy storage and
compare with the oracle under the tolerance of the contract.

Tolerance (per element, written here once and used by every parity test):
    |D - D_ref| <= 2^-7 * |alpha| * sum_k |a_ik||b_kj| + 1e-6   (BF16 / FP16)
    |D - D_ref| <= 2^-9 * |alpha| * sum_k |a_ik||b_kj| + 1e-6   (TF32)
D_ref and the scale come from the oracle in double.  Where D_ref is NaN the
kernel's value must be NaN too.
"""

from __future__ import annotations

import numpy as np

import seeded_inputs as si

TOL_REL = {"bf16": 2.0 ** -7, "fp16": 2.0 ** -7, "tf32": 2.0 ** -9}
TOL_ABS = 1e-6


def torch_storage(x: np.ndarray):
    """numpy storage -> CUDA torch tensor with the same bytes."""
    import torch

    if x.dtype == np.uint16:
        t = torch.from_numpy(x.view(np.int16).copy())
    else:
        t = torch.from_numpy(np.ascontiguousarray(x).copy())
    return t.cuda()


def run_tg(w: si.Workload, A: np.ndarray, B: np.ndarray, D0: np.ndarray | None = None,
           opts=None, stream=None, repeats: int = 1):
    """Launch tg_gemm(_ex) on copies of A, B and D0; return D storage (N, ldc)."""
    import torch
    import dense_gemm_epilogue_gb300 as tg

    lda, ldb, ldc = w.strides
    dA, dB = torch_storage(A), torch_storage(B)
    if D0 is None:
        D0 = si.make_output(w)
    dD = torch.from_numpy(np.ascontiguousarray(D0).copy()).cuda()
    outs = []
    for _ in range(repeats):
        if opts is None:
            st = tg.tg_gemm(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, dD, ldc, w.dtype,
                            w.relu, stream)
        else:
            st = tg.tg_gemm_ex(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, dD, ldc, w.dtype,
                               w.relu, opts, stream)
        tg.check(st)
        st, where = tg.tg_check_device_status(stream)
        assert st == tg.TG_OK, f"device status {st} at wait site {where}"
        outs.append(dD.cpu().numpy().copy())
    return outs if repeats > 1 else outs[0]


def logical(Dstore: np.ndarray, w: si.Workload) -> np.ndarray:
    """(N, ldc) storage -> logical (M, N) view."""
    return Dstore[:, : w.M].T


def assert_within(D: np.ndarray, ref: np.ndarray, scale: np.ndarray, dtype: str, what: str = ""):
    D = np.asarray(D, dtype=np.float64)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(D) & nan_ref, nan_ref), f"{what}: NaN positions differ"
    ok = ~nan_ref
    err = np.abs(D[ok] - ref[ok])
    bound = TOL_REL[dtype] * scale[ok] + TOL_ABS
    bad = ~(err <= bound)
    if bad.any():
        idx = np.flatnonzero(bad)[:8]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside tolerance; first "
            f"err={err[idx]}, bound={bound[idx]}, got={D[ok][idx]}, ref={ref[ok][idx]}")
    # The contract bound is loose; report the tighter relative error too.
    rel = err / np.maximum(scale[ok], 1e-30)
    return float(rel.max()) if rel.size else 0.0


def assert_padding_untouched(Dstore: np.ndarray, D0: np.ndarray, w: si.Workload):
    """Rows i >= M of every column (stride padding of D) keep their bytes."""
    got = Dstore[:, w.M:].view(np.uint32)
    want = D0[:, w.M:].view(np.uint32)
    assert np.array_equal(got, want), "D stride padding was written"


def check_full(w: si.Workload, opts=None, repeats: int = 1):
    """Whole-output parity of one workload against the oracle."""
    import oracle

    A, B = si.make_operands(w)
    lda, ldb, _ = w.strides
    D0 = si.make_output(w)
    out = run_tg(w, A, B, D0, opts=opts, repeats=repeats)
    outs = out if repeats > 1 else [out]
    ref, scale = oracle.gemm(w.M, w.N, w.K, w.alpha, A, lda, B, ldb, w.dtype, w.relu,
                             with_scale=True)
    rel = 0.0
    for o in outs:
        assert_padding_untouched(o, D0, w)
        rel = assert_within(logical(o, w), ref, scale, w.dtype, w.name)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32)), "not deterministic"
    return rel
