"""Plant a mistake in a copy of the oracle (on the CPU) and show that the pins
catch it: each mutant must fail at least one check of ``oracle_pin_checks``.

The mutants are the plausible slips: a dropped term, a wrong sign, a wrong
index or a transposed operand, a wrong exponent bias, a wrong tie rule, the
epilogue applied in the wrong order, and lost special values.
"""

import os

import pytest

import oracle
import oracle_pin_checks as pins

MUTANTS = {
    "drop_last_k": ("for (int64_t k = 0; k < jb->K; ++k) s += ai[k] * bj[k];",
                    "for (int64_t k = 0; k + 1 < jb->K; ++k) s += ai[k] * bj[k];"),
    "subtract_products": ("for (int64_t k = 0; k < jb->K; ++k) s += ai[k] * bj[k];",
                          "for (int64_t k = 0; k < jb->K; ++k) s -= ai[k] * bj[k];"),
    "reversed_k_in_A": ("Ad[i * K + k] = decode_elem(A, i * lda + k, dtype);",
                        "Ad[i * K + k] = decode_elem(A, i * lda + (K - 1 - k), dtype);"),
    "wrong_B_column": ("Bd[j * K + k] = decode_elem(B, k + j * ldb, dtype);",
                       "Bd[j * K + k] = decode_elem(B, k + (N - 1 - j) * ldb, dtype);"),
    "bf16_bias": ("v = ldexp((double)(128 + f), e - 127 - 7);",
                  "v = ldexp((double)(128 + f), e - 126 - 7);"),
    "fp16_subnormal_scale": ("v = ldexp((double)f, -14 - 10);",
                             "v = ldexp((double)f, -15 - 10);"),
    "tf32_ties_to_zero": ("if (r >= 0x1000u) q += 1;", "if (r > 0x1000u) q += 1;"),
    "tf32_truncate": ("if (r >= 0x1000u) q += 1;", "if (0) q += 1;"),
    "relu_keeps_negative_zero": ("return (y > 0.0) ? y : 0.0;", "return (y >= 0.0) ? y : 0.0;"),
    "relu_drops_nan": ("if (isnan(y)) return y;", "if (0) return y;"),
    "relu_before_alpha": ("double y = alpha * s;\n    return relu ? relu_max(y) : y;",
                          "return relu ? alpha * relu_max(s) : alpha * s;"),
    "alpha_dropped": ("double y = alpha * s;", "double y = s;"),
    "round_ties_away": ("if (r > 0.5 || (r == 0.5 && fmod(fq, 2.0) == 1.0)) fq += 1.0;",
                        "if (r >= 0.5) fq += 1.0;"),
    "round_no_overflow": ("if (out > maxf) out = INFINITY;", "if (0) out = INFINITY;"),
    "round_fp16_emin": ("case 2: y[q] = round_format(y[q], 11, -14, 15); break;",
                        "case 2: y[q] = round_format(y[q], 11, -15, 15); break;"),
    "e4m3_bias": ("else v = ldexp((double)(8 + f), e - 7 - 3);", "else v = ldexp((double)(8 + f), e - 8 - 3);"),
    "e4m3_subnormal": ("else if (e == 0) v = ldexp((double)f, -6 - 3);",
                       "else if (e == 0) v = ldexp((double)f, -7 - 3);"),
    "e4m3_no_nan": ("if (e == 0xF && f == 0x7) v = NAN;", "if (0) v = NAN;"),
    "e5m2_inf_as_nan": ("if (e == 0x1F) v = (f == 0) ? INFINITY : NAN;", "if (e == 0x1F) v = NAN;"),
    "e2m1_nibble_swap": ("return orc_decode_e2m1((idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF));",
                         "return orc_decode_e2m1((idx & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4));"),
    "e2m1_subnormal": ("double v = (e == 0) ? ldexp((double)f, -1)", "double v = (e == 0) ? ldexp((double)f, -2)"),
    "e2m1_bias": ("ldexp((double)(2 + f), e - 1 - 1);", "ldexp((double)(2 + f), e - 2 - 1);"),
    "epi_bias_row_by_column": ("case ORC_EPI_BIAS_ROW: return y + (double)bias[i];",
                               "case ORC_EPI_BIAS_ROW: return y + (double)bias[j];"),
    "epi_gelu_constant": ("(y + 0.044715 * y * y * y)", "(y + 0.04 * y * y * y)"),
    "epi_silu_as_sigmoid": ("case ORC_EPI_SILU: return y / (1.0 + exp(-y));",
                            "case ORC_EPI_SILU: return 1.0 / (1.0 + exp(-y));"),
    "epi_reverse_order": ("for (int q = 0; q < n_ops; ++q) y = apply_op(kinds[q], as[q], bs[q], biases[q], i, j, y);",
                          "for (int q = n_ops - 1; q >= 0; --q) y = apply_op(kinds[q], as[q], bs[q], biases[q], i, j, y);"),
    "epi_leaky_scales_positive": ("case ORC_EPI_LEAKY: return (isnan(y) || y > 0.0) ? y : a * y;",
                                  "case ORC_EPI_LEAKY: return a * y;"),
    "epi_clamp_bounds_swapped": ("        if (y < a) y = a;\n        if (y > b) y = b;",
                                 "        if (y < b) y = b;\n        if (y > a) y = a;"),
    "epi_alpha_after": ("int rc = orc_gemm(M, N, K, alpha, A, lda, B, ldb, dtype, 0, D, ldd, scale, nthreads);",
                        "int rc = orc_gemm(M, N, K, 1.0, A, lda, B, ldb, dtype, 0, D, ldd, scale, nthreads);"),
    "mx_block_16": ("#define ORC_MX_BLOCK 32", "#define ORC_MX_BLOCK 16"),
    "mx_block_64": ("#define ORC_MX_BLOCK 32", "#define ORC_MX_BLOCK 64"),
    "mx_scale_bias": ("return ldexp(1.0, (int)e - 127);", "return ldexp(1.0, (int)e - 128);"),
    "mx_scale_no_nan": ("if (e == 0xFF) return NAN;", "if (0) return NAN;"),
    "mx_only_a_scale": ("double x = xa[kb] * xb[kb];", "double x = xa[kb];"),
    "mx_block_shift": ("double x = xa[kb] * xb[kb];",
                       "double x = xa[kb] * xb[kb > 0 ? kb - 1 : 0];"),
    "mx_wrong_row_scale": ("(*Xa)[i * KB + kb] = scale_of(SA[i * ldsa + kb]);",
                           "(*Xa)[i * KB + kb] = scale_of(SA[(M - 1 - i) * ldsa + kb]);"),
    "nv_block_32": ("#define ORC_NV_BLOCK 16", "#define ORC_NV_BLOCK 32"),
    "nv_scales_as_exponents": ("ORC_E2M1,\n                       orc_decode_ue4m3, &Ad",
                               "ORC_E2M1,\n                       orc_decode_e8m0, &Ad"),
    "ue4m3_bias": ("return ldexp((double)(8 + m), e - 10);", "return ldexp((double)(8 + m), e - 11);"),
    "ue4m3_subnormal": ("if (e == 0) return ldexp((double)m, -9);",
                        "if (e == 0) return ldexp((double)m, -10);"),
    "ue4m3_no_nan": ("if (e == 15 && m == 7) return NAN;", "if (0) return NAN;"),
    "ue4m3_fraction_bits": ("return ldexp((double)(8 + m), e - 10);",
                            "return ldexp((double)(16 + m), e - 11);"),
    "nv_top_bit_accepted": ("if (SA[i * ldsa + kb] & 0x80) return -1;", "if (0) return -1;"),
    "mx_scale_abs_dropped": ("t += fabs(x) * bt;", "t += bt;"),
    "tf32_keeps_11_bits": ("uint32_t q = sig >> 13;           /* kept: 11 (or fewer) leading bits */\n"
                           "        uint32_t r = sig & 0x1FFFu;       /* dropped: 13 bits */\n"
                           "        if (r >= 0x1000u) q += 1;         /* half or more: away from zero */\n"
                           "        v = ldexp((double)q, ee - 23 + 13);",
                           "uint32_t q = sig >> 12;\n"
                           "        uint32_t r = sig & 0xFFFu;\n"
                           "        if (r >= 0x800u) q += 1;\n"
                           "        v = ldexp((double)q, ee - 23 + 12);"),
    "tf32_no_overflow": ("if (v > ldexp(2047.0, 127 - 10)) v = INFINITY;", "if (0) v = INFINITY;"),
    "bf16_subnormal_scale": ("v = ldexp((double)f, -126 - 7);", "v = ldexp((double)f, -127 - 7);"),
    "fp16_bias": ("v = ldexp((double)(1024 + f), e - 15 - 10);", "v = ldexp((double)(1024 + f), e - 14 - 10);"),
    "e5m2_bias": ("else v = ldexp((double)(4 + f), e - 15 - 2);", "else v = ldexp((double)(4 + f), e - 16 - 2);"),
    "lda_ignored": ("Ad[i * K + k] = decode_elem(A, i * lda + k, dtype);",
                    "Ad[i * K + k] = decode_elem(A, i * K + k, dtype);"),
    "ldb_ignored": ("Bd[j * K + k] = decode_elem(B, k + j * ldb, dtype);",
                    "Bd[j * K + k] = decode_elem(B, k + j * K, dtype);"),
    "epi_sigmoid_sign": ("case ORC_EPI_SIGMOID: return 1.0 / (1.0 + exp(-y));",
                         "case ORC_EPI_SIGMOID: return 1.0 / (1.0 + exp(y));"),
    "epi_bias_col_by_row": ("case ORC_EPI_BIAS_COL: return y + (double)bias[j];",
                            "case ORC_EPI_BIAS_COL: return y + (double)bias[i];"),
    "epi_add_subtracts": ("case ORC_EPI_ADD: return y + a;", "case ORC_EPI_ADD: return y - a;"),
    "round_bf16_extra_bit": ("case 1: y[q] = round_format(y[q], 8, -126, 127); break;",
                             "case 1: y[q] = round_format(y[q], 9, -126, 127); break;"),
    "round_no_subnormal_floor": ("if (ee < emin) ee = emin;", "if (0) ee = emin;"),
    "scale_signed_alpha": ("jb->scale[i + j * jb->ldd] = fabs(jb->alpha) * t;",
                           "jb->scale[i + j * jb->ldd] = jb->alpha * t;"),
}


def _run_checks(orc):
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.oracle.SOURCE) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / f"lib_{name}.so"))
    failed = _run_checks(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    lib = oracle.compile_source(oracle.oracle.SOURCE, str(tmp_path / "lib_ref.so"))
    assert _run_checks(oracle.Oracle(lib)) == []
    assert os.path.exists(lib)
