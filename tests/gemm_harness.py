"""Shared test plumbing: run tg_gemm through the C ABI on numpy storage and
compare with the oracle under the tolerance of the contract.

Tolerance (per element, written here once and used by every parity test):
    |D - D_ref| <= 2^-7 * |alpha| * sum_k |a_ik||b_kj| + 1e-6   (BF16 / FP16)
    |D - D_ref| <= 2^-9 * |alpha| * sum_k |a_ik||b_kj| + 1e-6   (TF32)
    |D - D_ref| <= 2^-7 * |alpha| * sum_k |a_ik||b_kj| + 1e-6   (E4M3 / E5M2)
D_ref and the scale come from the oracle in double.  Where D_ref is NaN the
kernel's value must be NaN too.  For the 8-bit floats the kernel reads the
same codes the oracle decodes and every product is exact in FP32 (4 x 4
significant bits at most), so only the FP32 accumulation differs: the 16-bit
kinds' bound applies unchanged.
"""

from __future__ import annotations

import numpy as np

import seeded_inputs as si

TOL_REL = {"bf16": 2.0 ** -7, "fp16": 2.0 ** -7, "tf32": 2.0 ** -9, "e4m3": 2.0 ** -7,
           "e5m2": 2.0 ** -7, "e2m1": 2.0 ** -7, "nvf4": 2.0 ** -7}
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


# ----------------------------------------------------------------- batched / narrow output

OUT_NP = {"f32": np.float32, "bf16": np.uint16, "fp16": np.uint16}
# Output rounding adds at most one unit in the last place of the output type.
OUT_ULP_REL = {"f32": 2.0 ** -23, "bf16": 2.0 ** -7, "fp16": 2.0 ** -10}
OUT_ULP_ABS = {"f32": 2.0 ** -149, "bf16": 2.0 ** -133, "fp16": 2.0 ** -24}


def decode_out(x: np.ndarray, out: str) -> np.ndarray:
    if out == "f32":
        return x.astype(np.float64)
    if out == "fp16":
        return x.view(np.float16).astype(np.float64)
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_batched(w: si.Workload, batch: int, out: str, share_a=False, share_b=False,
                pad_a=0, pad_b=0, pad_d=0, opts=None, repeats=1):
    """tg_gemm_batched on `batch` entries drawn with seeds w.seed, w.seed+1, ...
    Returns (A_list, B_list, D storage list per repeat, strides)."""
    import torch
    import dense_gemm_epilogue_gb300 as tg

    lda, ldb, ldc = w.strides
    entries = [si.make_operands(si.with_shape(w, seed=w.seed + b)) for b in range(batch)]
    A_list = [entries[0][0]] * batch if share_a else [e[0] for e in entries]
    B_list = [entries[0][1]] * batch if share_b else [e[1] for e in entries]
    sa = 0 if share_a else w.M * lda + pad_a
    sb = 0 if share_b else w.N * ldb + pad_b
    sd = w.N * ldc + pad_d
    ety = si.storage_numpy_dtype(w.dtype)
    A = np.zeros(max(sa * (batch - 1), 0) + w.M * lda, dtype=ety)
    B = np.zeros(max(sb * (batch - 1), 0) + w.N * ldb, dtype=ety)
    for b in range(batch):
        if not share_a or b == 0:
            A[b * sa: b * sa + w.M * lda] = A_list[b].reshape(-1)
        if not share_b or b == 0:
            B[b * sb: b * sb + w.N * ldb] = B_list[b].reshape(-1)
    sentinel = {"f32": np.uint32(0x7FC00002), "bf16": np.uint16(0x7FC3), "fp16": np.uint16(0x7E03)}
    D0 = np.full(sd * max(batch - 1, 0) + w.N * ldc, sentinel[out],
                 dtype=np.uint32 if out == "f32" else np.uint16)
    dA, dB = torch_storage(A), torch_storage(B)
    dD = torch.from_numpy(D0.view(np.int32 if out == "f32" else np.int16).copy()).cuda()
    outs = []
    for _ in range(repeats):
        st = tg.tg_gemm_batched(w.M, w.N, w.K, w.alpha, dA, lda, sa, dB, ldb, sb, dD, ldc, sd, batch,
                                w.dtype, out, w.relu, opts)
        tg.check(st, "tg_gemm_batched")
        st, where = tg.tg_check_device_status()
        assert st == tg.TG_OK, f"device status {st} at wait site {where}"
        outs.append(dD.cpu().numpy().view(np.uint32 if out == "f32" else np.uint16).copy())
    return A_list, B_list, D0, outs, (sa, sb, sd)


def check_batched(w: si.Workload, batch: int, out: str, repeats=1, **kw):
    import oracle

    lda, ldb, ldc = w.strides
    A_list, B_list, D0, outs, (sa, sb, sd) = run_batched(w, batch, out, repeats=repeats, **kw)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "not deterministic"
    Dall = outs[0]
    for b in range(batch):
        ref, scale = oracle.gemm(w.M, w.N, w.K, w.alpha, A_list[b], lda, B_list[b], ldb, w.dtype,
                                 w.relu, with_scale=True)
        ref_out = oracle.round_output(ref, out)
        store = Dall[b * sd: b * sd + w.N * ldc].reshape(w.N, ldc)
        got = decode_out(store[:, : w.M].view(OUT_NP[out]).T, out)
        # Stride padding of D (rows >= M, and the gap between batch entries) untouched.
        assert np.array_equal(store[:, w.M:], D0[b * sd: b * sd + w.N * ldc].reshape(w.N, ldc)[:, w.M:])
        if b + 1 < batch:
            gap = slice(b * sd + w.N * ldc, (b + 1) * sd)
            assert np.array_equal(Dall[gap], D0[gap])
        inf = np.isinf(ref_out)
        assert np.array_equal(got[inf], ref_out[inf]), f"{w.name}[{b}]: overflow differs"
        fin = ~inf
        tol = (TOL_REL[w.dtype] * scale + TOL_ABS + OUT_ULP_REL[out] * np.abs(ref) +
               OUT_ULP_ABS[out])
        nan_ref = np.isnan(ref_out)
        assert np.array_equal(np.isnan(got) & nan_ref, nan_ref)
        ok = fin & ~nan_ref
        err = np.abs(got[ok] - ref_out[ok])
        bad = ~(err <= tol[ok])
        if bad.any():
            i = np.flatnonzero(bad)[:6]
            raise AssertionError(f"{w.name}[{b}] ({out}): {bad.sum()} elements off; err={err[i]} "
                                 f"tol={tol[ok][i]} got={got[ok][i]} ref={ref_out[ok][i]}")


# ----------------------------------------------------------------- block-scaled (microscaling)

def to_atoms(S: np.ndarray, K: int, block: int = 32) -> np.ndarray:
    """Row-major scale codes (R, >= ceil(K/block)) -> the scale-atom byte
    layout of tg_gemm_mx: atom (rb, kg) at (rb * KG + kg) * 512, byte
    (r % 32) * 16 + ((r / 32) % 4) * 4 + kb % 4 inside it; zero padding."""
    R = S.shape[0]
    KB = -(-K // block)
    RB, KG = -(-R // 128), -(-KB // 4)
    full = np.zeros((RB * 128, KG * 4), dtype=np.uint8)
    full[:R, :KB] = S[:, :KB]
    # (rb, q, l, kg, j) with r = rb*128 + q*32 + l and kb = kg*4 + j
    t = full.reshape(RB, 4, 32, KG, 4)
    # atom (rb, kg), bytes in order (l, q, j)
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1)


def mx_padded(w: si.Workload):
    """The workload with lda, ldb rounded up to TMA-legal strides: multiples
    of 16 bytes (16 FP8 or 32 packed FP4 elements)."""
    q = 32 if w.dtype in ("e2m1", "nvf4") else 16
    rq = lambda x: -(-max(x, 1) // q) * q
    return si.with_shape(w, lda=w.lda or rq(w.K), ldb=w.ldb or rq(w.K))


def run_mx(w: si.Workload, A, B, SA, SB, out="f32", opts=None, repeats=1, D0=None):
    """tg_gemm_mx on the given storage (A (M, lda), B (N, ldb) FP8 codes,
    SA (M, KB), SB (N, KB) row-major scale codes).  Returns D storage (N, ldc)
    per repeat."""
    import torch
    import dense_gemm_epilogue_gb300 as tg

    lda, ldb, ldc = w.strides
    dA, dB = torch_storage(A), torch_storage(B)
    blk = si.scale_block(w.dtype)
    dSA = torch_storage(to_atoms(SA, w.K, blk))
    dSB = torch_storage(to_atoms(SB, w.K, blk))
    assert dSA.numel() == tg.tg_bs_scale_bytes(w.M, w.K, w.dtype)
    assert dSB.numel() == tg.tg_bs_scale_bytes(w.N, w.K, w.dtype)
    onp = {"f32": np.uint32, "bf16": np.uint16, "fp16": np.uint16}[out]
    if D0 is None:
        D0 = np.full((w.N, ldc), 0x7FC00002 if out == "f32" else 0x7FC3, dtype=onp)
    tdt = torch.int32 if out == "f32" else torch.int16
    dD = torch.from_numpy(D0.view(np.int32 if out == "f32" else np.int16).copy()).cuda()
    outs = []
    for _ in range(repeats):
        st = tg.tg_gemm_mx(w.M, w.N, w.K, w.alpha, dA, lda, dSA, dB, ldb, dSB, dD, ldc, w.dtype,
                           out, w.relu, opts)
        tg.check(st, "tg_gemm_mx")
        st, where = tg.tg_check_device_status()
        assert st == tg.TG_OK, f"device status {st} at wait site {where}"
        outs.append(dD.cpu().numpy().view(onp).copy())
    assert tdt is not None
    return D0, outs


def check_mx(w: si.Workload, out="f32", opts=None, repeats=1, scale_range=None):
    """Whole-output parity of tg_gemm_mx against the oracle's block-scaled
    product: |D - D_ref| <= 2^-7 * |alpha| * sum_kb |Xa Xb| sum |a||b| + 1e-6
    (plus one output ulp for narrow outputs); padding untouched; repeats
    bitwise identical.  Returns the largest error relative to that scale."""
    import oracle

    w = mx_padded(w)
    lda, ldb, ldc = w.strides
    A, B = si.make_operands(w)
    SA, SB = si.make_mx_scales(w, *(scale_range or (None, None)))
    D0, outs = run_mx(w, A, B, SA, SB, out=out, opts=opts, repeats=repeats)
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "not deterministic"
    KB = -(-w.K // si.scale_block(w.dtype))
    ref, scale = oracle.gemm_mx(w.M, w.N, w.K, w.alpha, A, lda, SA, max(KB, 1), B, ldb, SB,
                                max(KB, 1), w.dtype, w.relu, with_scale=True)
    store = outs[0]
    assert np.array_equal(store[:, w.M:], D0[:, w.M:]), "D stride padding was written"
    got = decode_out(store[:, : w.M].view(OUT_NP[out]).T, out)
    ref_out = oracle.round_output(ref, out)
    nan_ref = np.isnan(ref_out)
    assert np.array_equal(np.isnan(got) & nan_ref, nan_ref), f"{w.name}: NaN positions differ"
    inf = np.isinf(ref_out)
    assert np.array_equal(got[inf], ref_out[inf]), f"{w.name}: overflow differs"
    ok = ~nan_ref & ~inf
    err = np.abs(got[ok] - ref_out[ok])
    tol = TOL_REL[w.dtype] * scale[ok] + TOL_ABS
    if out != "f32":
        tol = tol + OUT_ULP_REL[out] * np.abs(ref[ok]) + OUT_ULP_ABS[out]
    bad = ~(err <= tol)
    if bad.any():
        idx = np.flatnonzero(bad)[:8]
        raise AssertionError(f"{w.name}: {bad.sum()} of {bad.size} elements off; err={err[idx]} "
                             f"tol={tol[idx]} got={got[ok][idx]} ref={ref_out[ok][idx]}")
    rel = err / np.maximum(scale[ok], 1e-30)
    return float(rel.max()) if rel.size else 0.0


# ----------------------------------------------------------------- composed pointwise epilogues

# Largest slope of each op (how much it can grow an error in its input).
EPI_LIPSCHITZ = {"scale": None, "add": 1.0, "relu": 1.0, "leaky_relu": None, "clamp": 1.0,
                 "sigmoid": 0.25, "silu": 1.1, "gelu_tanh": 1.13, "bias_row": 1.0, "bias_col": 1.0}


def epi_lipschitz(ops) -> float:
    lip = 1.0
    for kind, a, _b, _bias in ops:
        if kind == "scale":
            lip *= abs(a)
        elif kind == "leaky_relu":
            lip *= max(1.0, abs(a))
        else:
            lip *= EPI_LIPSCHITZ[kind]
    return lip


def check_epi(w: si.Workload, ops, out="f32", opts=None, repeats=1, bias_seed=5):
    """tg_gemm_epilogue against the oracle's composed epilogue, every element:
    |D - D_ref| <= TOL_REL * |alpha| sum|a||b| * L + 2^-18 (1 + |D_ref|) + 1e-6
    (+ one output ulp), L the product of the ops' largest slopes (the GEMM
    bound carried through the chain) and the 2^-18 term the FP32 evaluation of
    the ops.  `ops` use names; a bias entry of "rows" / "cols" is replaced by
    a seeded float32 vector of M / N values.  D's stride padding must be
    untouched; repeats bitwise identical."""
    import torch
    import oracle
    import dense_gemm_epilogue_gb300 as tg

    lda, ldb, ldc = w.strides
    A, B = si.make_operands(w)
    host_ops, dev_ops, keep = [], [], []
    for q, (kind, a, b, bias) in enumerate(ops):
        vec = None
        if bias in ("rows", "cols"):
            n = w.M if bias == "rows" else w.N
            vec = si.uniform_f32(bias_seed, 10 + q, n, -1.0, 1.0).astype(np.float32)
            t = torch.from_numpy(vec).cuda()
            keep.append(t)
        host_ops.append((kind, a, b, vec))
        dev_ops.append((kind, a, b, keep[-1] if vec is not None else None))
    onp = {"f32": np.uint32, "bf16": np.uint16, "fp16": np.uint16}[out]
    D0 = np.full((w.N, ldc), 0x7FC00002 if out == "f32" else 0x7FC3, dtype=onp)
    dA, dB = torch_storage(A), torch_storage(B)
    dD = torch.from_numpy(D0.view(np.int32 if out == "f32" else np.int16).copy()).cuda()
    outs = []
    for _ in range(repeats):
        st = tg.tg_gemm_epilogue(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, dD, ldc, w.dtype, out,
                                 dev_ops, opts)
        tg.check(st, "tg_gemm_epilogue")
        st, where = tg.tg_check_device_status()
        assert st == tg.TG_OK, f"device status {st} at wait site {where}"
        outs.append(dD.cpu().numpy().view(onp).copy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "not deterministic"
    ref, scale = oracle.gemm_epi(w.M, w.N, w.K, w.alpha, A, lda, B, ldb, w.dtype, host_ops,
                                 with_scale=True)
    store = outs[0]
    assert np.array_equal(store[:, w.M:], D0[:, w.M:]), "D stride padding was written"
    got = decode_out(store[:, : w.M].view(OUT_NP[out]).T, out)
    ref_out = oracle.round_output(ref, out)
    nan_ref = np.isnan(ref_out)
    assert np.array_equal(np.isnan(got) & nan_ref, nan_ref), f"{w.name}: NaN positions differ"
    ok = ~nan_ref
    err = np.abs(got[ok] - ref_out[ok])
    tol = (TOL_REL[w.dtype] * scale[ok] * epi_lipschitz(ops) + 2.0 ** -18 * (1 + np.abs(ref[ok]))
           + TOL_ABS)
    if out != "f32":
        tol = tol + OUT_ULP_REL[out] * np.abs(ref[ok]) + OUT_ULP_ABS[out]
    bad = ~(err <= tol)
    if bad.any():
        idx = np.flatnonzero(bad)[:8]
        raise AssertionError(f"{w.name} {ops}: {bad.sum()} of {bad.size} off; err={err[idx]} "
                             f"tol={tol[idx]} got={got[ok][idx]} ref={ref_out[ok][idx]}")


# ----------------------------------------------------------------- batched block-scaled

def _bias_vectors(w: si.Workload, ops, bias_seed: int):
    """Ops with "rows" / "cols" bias entries replaced by seeded float32
    vectors of M / N values: (host ops, device ops, device tensors kept)."""
    import torch

    host_ops, dev_ops, keep = [], [], []
    for q, (kind, a, b, bias) in enumerate(ops):
        vec = None
        if bias in ("rows", "cols"):
            n = w.M if bias == "rows" else w.N
            vec = si.uniform_f32(bias_seed, 10 + q, n, -1.0, 1.0).astype(np.float32)
            keep.append(torch.from_numpy(vec).cuda())
        host_ops.append((kind, a, b, vec))
        dev_ops.append((kind, a, b, keep[-1] if vec is not None else None))
    return host_ops, dev_ops, keep


def check_mx_batched(w: si.Workload, batch: int, out="f32", ops=(), share_a=False, share_b=False,
                     share_sfa=False, share_sfb=False, pad_a=0, pad_b=0, pad_sf=0, pad_d=0,
                     opts=None, repeats=1, scale_range=None, bias_seed=7):
    """tg_gemm_mx_batched on `batch` entries drawn with seeds w.seed, w.seed+1,
    ... (operands and scales each either per entry or shared), against the
    oracle's block-scaled product of each entry followed by its op chain,
    every element, with check_epi's bound.  Operand paddings count elements
    (multiples of 16 bytes); pad_sf counts bytes.  D's padding and the gaps
    between entries must be untouched; repeats bitwise identical."""
    import torch
    import oracle
    import dense_gemm_epilogue_gb300 as tg

    w = mx_padded(w)
    lda, ldb, ldc = w.strides
    per = 2 if w.dtype in ("e2m1", "nvf4") else 1  # elements per storage byte
    blk = si.scale_block(w.dtype)
    KB = -(-w.K // blk)
    ents = [si.with_shape(w, seed=w.seed + b) for b in range(batch)]
    ops_ = [si.make_operands(e) for e in ents]
    scs = [si.make_mx_scales(e, *(scale_range or (None, None))) for e in ents]
    pick = lambda lst, shared: [lst[0]] * batch if shared else lst
    A_list = pick([o[0] for o in ops_], share_a)
    B_list = pick([o[1] for o in ops_], share_b)
    SA_list = pick([s[0] for s in scs], share_sfa)
    SB_list = pick([s[1] for s in scs], share_sfb)
    sa = 0 if share_a else w.M * lda + pad_a
    sb = 0 if share_b else w.N * ldb + pad_b
    fa, fb = tg.tg_bs_scale_bytes(w.M, w.K, w.dtype), tg.tg_bs_scale_bytes(w.N, w.K, w.dtype)
    ssa = 0 if share_sfa else fa + pad_sf
    ssb = 0 if share_sfb else fb + pad_sf
    sd = w.N * ldc + pad_d

    def pack(lst, stride_bytes, one_bytes, dtype):
        buf = np.zeros(max(stride_bytes * (batch - 1), 0) + one_bytes, dtype=dtype)
        for b in range(batch if stride_bytes else 1):
            buf[b * stride_bytes: b * stride_bytes + one_bytes] = lst[b].reshape(-1)
        return buf

    ety = A_list[0].dtype
    A = pack(A_list, sa // per, A_list[0].size, ety)
    B = pack(B_list, sb // per, B_list[0].size, ety)
    SA = pack([to_atoms(s, w.K, blk) for s in SA_list], ssa, fa, np.uint8)
    SB = pack([to_atoms(s, w.K, blk) for s in SB_list], ssb, fb, np.uint8)
    host_ops, dev_ops, keep = _bias_vectors(w, ops, bias_seed)
    sentinel = {"f32": np.uint32(0x7FC00002), "bf16": np.uint16(0x7FC3), "fp16": np.uint16(0x7E03)}
    onp = np.uint32 if out == "f32" else np.uint16
    D0 = np.full(sd * max(batch - 1, 0) + w.N * ldc, sentinel[out], dtype=onp)
    dev = lambda x: torch_storage(x) if x.size else None
    dA, dB, dSA, dSB = dev(A), dev(B), dev(SA), dev(SB)
    dD = torch.from_numpy(D0.view(np.int32 if out == "f32" else np.int16).copy()).cuda()
    outs = []
    for _ in range(repeats):
        st = tg.tg_gemm_mx_batched(w.M, w.N, w.K, w.alpha, dA, lda, sa, dSA, ssa, dB, ldb, sb,
                                   dSB, ssb, dD, ldc, sd, batch, w.dtype, out, dev_ops, opts)
        tg.check(st, "tg_gemm_mx_batched")
        st, where = tg.tg_check_device_status()
        assert st == tg.TG_OK, f"device status {st} at wait site {where}"
        outs.append(dD.cpu().numpy().view(onp).copy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "not deterministic"
    Dall = outs[0]
    lip = epi_lipschitz(ops)
    worst = 0.0
    for b in range(batch):
        prod, scale = oracle.gemm_mx(w.M, w.N, w.K, w.alpha, A_list[b], lda, SA_list[b],
                                     max(KB, 1), B_list[b], ldb, SB_list[b], max(KB, 1), w.dtype,
                                     False, with_scale=True)
        ref = oracle.apply_epi(prod, host_ops)
        ref_out = oracle.round_output(ref, out)
        store = Dall[b * sd: b * sd + w.N * ldc].reshape(w.N, ldc)
        pad0 = D0[b * sd: b * sd + w.N * ldc].reshape(w.N, ldc)
        assert np.array_equal(store[:, w.M:], pad0[:, w.M:]), "D stride padding was written"
        if b + 1 < batch:
            gap = slice(b * sd + w.N * ldc, (b + 1) * sd)
            assert np.array_equal(Dall[gap], D0[gap]), "gap between entries was written"
        got = decode_out(store[:, : w.M].view(OUT_NP[out]).T, out)
        nan_ref = np.isnan(ref_out)
        assert np.array_equal(np.isnan(got) & nan_ref, nan_ref), f"{w.name}[{b}]: NaN positions"
        inf = np.isinf(ref_out)
        assert np.array_equal(got[inf], ref_out[inf]), f"{w.name}[{b}]: overflow differs"
        ok = ~nan_ref & ~inf
        err = np.abs(got[ok] - ref_out[ok])
        tol = TOL_REL[w.dtype] * scale[ok] * lip + 2.0 ** -18 * (1 + np.abs(ref[ok])) + TOL_ABS
        if out != "f32":
            tol = tol + OUT_ULP_REL[out] * np.abs(ref[ok]) + OUT_ULP_ABS[out]
        bad = ~(err <= tol)
        if bad.any():
            idx = np.flatnonzero(bad)[:8]
            raise AssertionError(f"{w.name}[{b}] {ops}: {bad.sum()} of {bad.size} off; "
                                 f"err={err[idx]} tol={tol[idx]} got={got[ok][idx]} "
                                 f"ref={ref_out[ok][idx]}")
        if err.size:
            worst = max(worst, float((err / np.maximum(scale[ok], 1e-30)).max()))
    del keep
    return worst
