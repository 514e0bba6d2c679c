"""The hand-worked examples of tests/golden/hand_examples.json through the
CUDA path.  Every entry is exactly representable in its storage type and
every product and sum is exact in FP32, so the kernel's D must equal the
worked values exactly.  On the GPU this pins what the parity tolerance alone
cannot tell apart: alpha applied before the max with zero ("Walk through
GEMM", section 5) and the TF32 narrowing's tie rule (round to nearest, ties
away from zero; "Matrix Multiplication", Step 4).  Each case runs with tight
strides (plain-load producer) and with rows padded to 16 bytes (TMA), the
padding filled with NaN, which must never be read; D's stride padding must
stay untouched."""

from __future__ import annotations

import json
import os

import numpy as np
import pytest

import oracle_pin_checks as pins
from gemm_harness import torch_storage

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_examples.json")
with open(GOLDEN) as _f:
    CASES = json.load(_f)["cases"]
ELEM = {"bf16": 2, "fp16": 2, "tf32": 4}


@pytest.fixture(scope="module")
def tg():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()
    return tg


@pytest.mark.parametrize("strides", ["tight", "padded"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_worked_example_is_exact(tg, case, strides):
    import torch

    dtype = case["dtype"]
    Alog = np.asarray(case["A"], dtype=np.float64)
    Blog = np.asarray(case["B"], dtype=np.float64)
    M, K = Alog.shape
    N = Blog.shape[1]
    per16 = 16 // ELEM[dtype]
    ld = K if strides == "tight" else -(-K // per16) * per16 + per16
    A, lda, B, ldb = pins.pack(Alog, Blog, dtype, ld, ld)
    ldc = M + 3
    D0 = np.full((N, ldc), 0x7FC00002, dtype=np.uint32).view(np.float32)
    dA, dB = torch_storage(A), torch_storage(B)
    dD = torch.from_numpy(D0.copy()).cuda()
    plan = tg.tg_plan(M, N, K, dA, lda, dB, ldb, dD, ldc, dtype)
    assert plan["producer"] == (1 if strides == "padded" else 2)
    tg.check(tg.tg_gemm(M, N, K, case["alpha"], dA, lda, dB, ldb, dD, ldc, dtype, case["relu"]))
    st, where = tg.tg_check_device_status(None)
    assert st == tg.TG_OK, f"device status {st} at wait site {where}"
    out = dD.cpu().numpy()
    got = out[:, :M].T.astype(np.float64)
    want = np.asarray(case["D"], dtype=np.float64)
    assert np.array_equal(got, want), (case["name"], got, want)
    assert np.array_equal(out[:, M:].view(np.uint32), D0[:, M:].view(np.uint32))
