"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is a textual edit of a copy of the oracle's C source, compiled on
the CPU into a temporary library; the pins of ``oracle_pins`` then run
against it.  A mutant that no pin rejects means the pins cannot tell that
mistake from the contract.  The first three are the defects the case study
"Aligning fused RMSNorm rounding across vLLM backends" discusses (early
rounding of the sum, and the two wrong orders of the weighted-output cast);
the rest are the slips a plain implementation could make.
"""
import os

import pytest

import oracle
import oracle_pins as P

SRC = open(oracle.SOURCE).read()

MUTANTS = {
    # the early-rounding defect: variance and normalisation from the rounded sum
    "early_rounding": [("s[i] = xf + rf;", "s[i] = round_to(act, xf + rf);")],
    # cast to the activation dtype instead of the weight dtype
    "cast_to_act": [("float n = round_to(wd, a);               /* weight dtype first */",
                     "float n = round_to(act, a);")],
    # multiply by the weight before casting
    "multiply_then_cast": [("float n = round_to(wd, a);               /* weight dtype first */", "float n = a;")],
    "divisor_h_minus_1": [("float var = S / (float)hidden;",
                           "float var = S / (float)(hidden > 1 ? hidden - 1 : 1);")],
    "eps_dropped": [("float var = S / (float)hidden;\n    float tv = var + eps;",
                     "float var = S / (float)hidden;\n    float tv = var;")],
    "eps_outside_root": [("float var = S / (float)hidden;\n    float tv = var + eps;",
                          "float var = S / (float)hidden;\n    float tv = var;"),
                         ("float rstd = 1.0f / root;", "float rstd = 1.0f / root + eps;")],
    "abs_not_square": [("float sq = s[i] * s[i];", "float sq = fabsf(s[i]);")],
    "weight_index_shift": [("float prod = n * load(weight, wd, i);",
                            "float prod = n * load(weight, wd, (i + 1) % hidden);")],
    "residual_unrounded_store": [("/* binary32 add, kept unrounded */\n                store(rorow, act, i, round_to(act, s[i]));",
                                  "/* binary32 add, kept unrounded */\n                store(rorow, act, i, s[i]);")],
    "residual_reads_x_twice": [("float rf = load(rr, act, i);", "float rf = load(xr, act, i);")],
    "negated_output": [("float a = s[i] * rstd;", "float a = -s[i] * rstd;")],
    "ties_away_from_zero": [("if (rest > half || (rest == half && (keep & 1u))) keep += 1;",
                             "if (rest >= half) keep += 1;")],
    "sum_truncated": [("if (guard && (sticky || (keep & 1u))) keep += 1;", "")],
    "sum_sequential_binary32": [("float S = acc_round(&acc);",
                                 "float S = 0.0f; for (int64_t i = 0; i < hidden; ++i) S += s[i] * s[i];")],
    "rstd_single_rounding": [("float root = sqrtf(tv);\n    float rstd = 1.0f / root;",
                              "float root = sqrtf(tv);\n    float rstd = (float)(1.0 / sqrt((double)tv));")],
    # (these two sites recur in the LayerNorm driver, which gets the same slip)
    "out_row_stride_of_act": [("char* orow = (char*)out + (size_t)t * (size_t)hidden * so;",
                               "char* orow = (char*)out + (size_t)t * (size_t)hidden * sa;", "all")],
    "no_residual_doubles_x": [("                s[i] = xf;\n", "                s[i] = xf + xf;\n", "all")],
    "f16_subnormal_encoding": [("return (uint16_t)(sign | (uint16_t)(m >> (-e - 1)));",
                                "return (uint16_t)(sign | (uint16_t)(m >> (-e)));")],
    # (">" instead of ">=" here would be an equivalent mutant: a value rounded to
    # exactly 2^16 encodes as the fp16 infinity anyway, and no |a| reaches it)
    "overflow_exponent_off_by_one": [("if (mag >= ldexp(1.0, emax + 1)) mag = INFINITY;\n    float r = (float)mag;",
                                      "if (mag >= ldexp(1.0, emax)) mag = INFINITY;\n    float r = (float)mag;")],
}


@pytest.fixture(scope="module")
def cases():
    return P.pin_cases()


def _mutant_lib(tmp_path, name, edits):
    src = SRC
    for old, new, *scope in edits:
        n = src.count(old)
        assert n == 1 or (scope == ["all"] and n >= 1), f"mutant {name}: edit site not unique/found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    return oracle.bind(oracle.compile_oracle(str(path), str(tmp_path / f"lib{name}.so")))


def _failed_pins(L, cases):
    failed = []
    for pin in P.ALL_PINS:
        try:
            if pin in (P.pin_policy, P.pin_closed_forms):
                pin(L)
            else:
                pin(L, cases)
        except AssertionError:
            failed.append(pin.__name__)
        except (RuntimeError, ValueError):
            failed.append(pin.__name__ + "(error)")
    return failed


def _extra_pin_checks(L):
    """Converter pins on boundary values (the exhaustive sweep lives in its own test)."""
    import test_oracle_converters as C
    failed = []
    for check in (C.check_page_format_facts, C.check_converter_boundaries):
        try:
            check(L)
        except AssertionError:
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, cases, name):
    L = _mutant_lib(tmp_path, name, MUTANTS[name])
    failed = _failed_pins(L, cases) + _extra_pin_checks(L)
    assert failed, f"no pin rejects the planted mistake {name!r}"


@pytest.mark.parametrize("name", ["rstd_single_rounding", "eps_outside_root", "eps_dropped", "early_rounding"])
def test_exhaustive_hidden_1_catches(tmp_path, name):
    """The exhaustive hidden = 1 sweep alone rejects mistakes in the rstd step (and the
    early rounding of the sum); the unmutated copy passes it."""
    L = _mutant_lib(tmp_path, name, MUTANTS[name])
    with pytest.raises(AssertionError):
        P.pin_exhaustive_h1(L)


def test_exhaustive_hidden_1_passes_the_unmutated_copy(tmp_path):
    P.pin_exhaustive_h1(_mutant_lib(tmp_path, "identity_h1", []))


def test_unmutated_copy_passes(tmp_path, cases):
    L = _mutant_lib(tmp_path, "identity", [])
    assert _failed_pins(L, cases) == []
    assert _extra_pin_checks(L) == []


QUANT_MUTANTS = {
    # the maximum without the absolute value
    "amax_signed": [("float a = fabsf(o[i]);", "float a = o[i];")],
    # divisor 128 instead of the symmetric 127
    "int8_divisor_128": [("const float qmax = qtype == OR_Q_INT8 ? 127.0f : 448.0f;",
                          "const float qmax = qtype == OR_Q_INT8 ? 128.0f : 448.0f;")],
    # truncation instead of rounding to nearest
    "int8_truncates": [("if (d > 0.5f || (d == 0.5f && fmodf(f, 2.0f) != 0.0f)) n = f + 1.0f;", "")],
    # ties away from zero
    "int8_ties_away": [("if (d > 0.5f || (d == 0.5f && fmodf(f, 2.0f) != 0.0f)) n = f + 1.0f;",
                        "if (d >= 0.5f) n = f + 1.0f;")],
    # quantising the binary32 product instead of the stored out value: scale from s * rstd
    "quantise_normalised_not_out": [("for (int64_t i = 0; i < hidden; ++i) of[i] = load(orow, od, i);",
                                     "for (int64_t i = 0; i < hidden; ++i) of[i] = load(orow, od, i) * 1.001f;")],
    # E4M3 without saturation: the top code becomes 480 (a NaN code)
    "e4m3_no_saturation": [("if (r > 448.0f) r = 448.0f;", "")],
    # E4M3 exponent bias off by one
    "e4m3_bias": [("return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)((m >> 20) & 0x7u));",
                   "return (uint8_t)(sign | (uint8_t)((e + 8) << 3) | (uint8_t)((m >> 20) & 0x7u));")],
    # scale = QMAX / amax (the inverse stored instead of the scale)
    "scale_inverted": [("    return scale;\n}", "    return inv;\n}")],
}


@pytest.mark.parametrize("name", sorted(QUANT_MUTANTS))
def test_quant_mutant_is_caught(tmp_path, name):
    import test_oracle_quant as TQ
    L = _mutant_lib(tmp_path, name, QUANT_MUTANTS[name])
    failed = []
    for check in (TQ.check_e4m3_format, TQ.check_int8, TQ.check_quant_rows):
        try:
            check(L)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no quant pin rejects the planted mistake {name!r}"


def test_unmutated_copy_passes_quant_pins(tmp_path):
    import test_oracle_quant as TQ
    L = _mutant_lib(tmp_path, "identity_q", [])
    for check in (TQ.check_e4m3_format, TQ.check_int8, TQ.check_quant_rows):
        check(L)


LN_MUTANTS = {
    # the "Mixed-Precision Kernels" page's one-pass sketch: var = E[s^2] - mean^2
    "one_pass_variance": [("        d[i] = s[i] - mean;\n        float sq = d[i] * d[i];",
                           "        d[i] = s[i] - mean;\n        float sq = s[i] * s[i];"),
                          ("    float var = S2 / (float)hidden;\n    float tv = var + eps;",
                           "    float var = S2 / (float)hidden - mean * mean;\n    float tv = var + eps;")],
    "mean_over_h_minus_1": [("    float mean = S1 / (float)hidden;",
                             "    float mean = S1 / (float)(hidden > 1 ? hidden - 1 : 1);")],
    "beta_before_cast": [("            float n = round_to(wd, a);                  /* weight dtype first */",
                          "            float n = round_to(wd, a + load(beta, wd, i) / load(gamma, wd, i));")],
    "no_weight_cast_ln": [("            float n = round_to(wd, a);                  /* weight dtype first */",
                           "            float n = a;")],
    "beta_dropped": [("            float u = t1 + load(beta, wd, i);           /* ... and the shift */",
                      "            float u = t1;")],
    "signed_sum_drops_negatives": [("    else if (v < 0) acc_add(&a->neg, -v);", "")],
    "ln_eps_dropped": [("    float tv = var + eps;\n    float root = sqrtf(tv);\n    if (mean_out)",
                        "    float tv = var;\n    float root = sqrtf(tv);\n    if (mean_out)")],
}


@pytest.mark.parametrize("name", sorted(LN_MUTANTS))
def test_layernorm_mutant_is_caught(tmp_path, name):
    import test_oracle_layernorm as TL
    L = _mutant_lib(tmp_path, name, LN_MUTANTS[name])
    failed = []
    for check in (TL.check_signed_sum, TL.check_steps, TL.check_closed_forms, TL.check_fp64):
        try:
            check(L)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no LayerNorm pin rejects the planted mistake {name!r}"


def test_unmutated_copy_passes_layernorm_pins(tmp_path):
    import test_oracle_layernorm as TL
    L = _mutant_lib(tmp_path, "identity_ln", [])
    for check in (TL.check_signed_sum, TL.check_steps, TL.check_closed_forms, TL.check_fp64):
        check(L)


GEMM_MUTANTS = {
    # the page's rejected implementation: products rounded to fp16 before the sum
    "gemm_products_rounded_to_f16": [("sacc_add(&acc, a * b);   /* exact: see above */",
                                      "sacc_add(&acc, round_f16(a * b));")],
    # the sum rounded to binary32 first, then to fp16 (double rounding)
    "gemm_cast_through_f32": [("double p16 = sacc_round_format(&acc, 11, -14, 15);",
                               "double p16 = round_double_f16((double)sacc_round(&acc));")],
    # the bias added to the unrounded sum (across the projection's rounding boundary)
    "gemm_bias_before_cast": [("double p16 = sacc_round_format(&acc, 11, -14, 15);",
                               "if (bias) sacc_add(&acc, decode_f16(bias[n]));\n"
                               "            double p16 = sacc_round_format(&acc, 11, -14, 15);"),
                              ("double y = bias ? round_double_f16(p16 + (double)decode_f16(bias[n])) : p16;",
                               "double y = p16;")],
    # the weight read as [K, N] instead of the transposed [N, K] (kept in bounds)
    "gemm_weight_not_transposed": [("float b = decode_f16(wt[n * K + k]);",
                                    "float b = decode_f16(wt[(k * N + n) % (N * K)]);")],
    # ties away from zero in the fp16 cast of the sum
    "gemm_ties_away": [("if (kq > 0 && guard && (sticky || (keep & 1u))) keep += 1;",
                        "if (kq > 0 && guard) keep += 1;")],
    # (dropping the overflow test of the cast would be an equivalent mutant: a sum that
    # rounds to 2^16 encodes as the fp16 infinity anyway, and no binary32 sum of fp16
    # products reaches 2^128)
}


@pytest.mark.parametrize("name", sorted(GEMM_MUTANTS))
def test_gemm_mutant_is_caught(tmp_path, name):
    import test_oracle_gemm as TG
    L = _mutant_lib(tmp_path, name, GEMM_MUTANTS[name])
    failed = []
    for check in TG.GEMM_CHECKS:
        try:
            check(L)
        except (AssertionError, RuntimeError):
            failed.append(check.__name__)
    assert failed, f"no pin rejects the planted mistake {name!r}"
