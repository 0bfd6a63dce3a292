"""The oracle's pins catch plausible mistakes in it.

Each case below plants one mistake in a copy of the oracle's C source (never
in the committed file), compiles the copy on the CPU, loads it as a separate
oracle module and runs a chosen set of the pins from ``test_oracle_amsim`` and
``test_oracle_contractions`` against it: at least one of them must fail.  The
mistakes are the kinds a restatement of Algorithms 1-2 (ApproxTrain Sec. V-A,
V-B) and of the convolution sums (Sec. VI-B, Algorithms 3-4; depthwise from
Sec. III, Table I) is likely to contain: an exponent bias, a dropped carry, the
zero test's boundary, Mitchell's branch, truncation vs rounding, denormals,
transposes, dilation and flip indices, channel-multiplier indexing, the
tolerance scale, a user table's index order and carry, Algorithm 1's carry
detection over a user model, and the exponent cast of (1, e, m) formats.
"""
import importlib.util
import os
import re
import shutil

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "amsim_oracle.c")


def _load_test_module(name):
    spec = importlib.util.spec_from_file_location(f"_mut_{name}", os.path.join(HERE, f"{name}.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


T_AMSIM = _load_test_module("test_oracle_amsim")
T_CONTR = _load_test_module("test_oracle_contractions")
T_USER = _load_test_module("test_oracle_usermodels")
T_FMT = _load_test_module("test_oracle_formats")


def _function_span(src, fname):
    """[start, end) of the definition of C function `fname` (to its closing brace
    at column 0)."""
    m = re.search(r"^[a-z].*\b" + re.escape(fname) + r"\(", src, re.M)
    assert m, fname
    end = src.index("\n}\n", m.start()) + 3
    return m.start(), end


def _mutant_oracle(tmp_path, fname, old, new):
    src = open(SRC).read()
    a, b = _function_span(src, fname)
    body = src[a:b]
    assert body.count(old) == 1, (fname, old)
    src = src[:a] + body.replace(old, new) + src[b:]
    d = tmp_path / "oracle"
    d.mkdir()
    (d / "amsim_oracle.c").write_text(src)
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), d / "__init__.py")
    spec = importlib.util.spec_from_file_location(f"_mut_oracle_{tmp_path.name}", str(d / "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.lib()   # compiles the copy into its own _build directory
    return mod


def _dw_geom(i):
    return T_CONTR.DW_GEOMS[i]


# name: (function, old text, new text, pins that should catch it)
MUTANTS = {
    "exponent_bias": ("algorithm2", "int e0 = ea + eb - bias;", "int e0 = ea + eb - bias + 1;",
                      [T_AMSIM.test_special_values_hand_worked, T_AMSIM.test_mitchell_scaling_in_normal_range]),
    "dropped_carry": ("algorithm2", "int e = e0 + (int)carry;", "int e = e0;",
                      [T_AMSIM.test_mitchell_hand_values, T_AMSIM.test_mitchell_scaling_in_normal_range]),
    "zero_test_boundary": ("algorithm2", "if (e0 <= 0) return s << 31;", "if (e0 < 0) return s << 31;",
                           [T_AMSIM.test_special_values_hand_worked]),
    "zero_test_after_carry": ("algorithm2", "if (e0 <= 0) return s << 31;",
                              "if (e0 + (int)carry <= 0) return s << 31;",
                              [T_AMSIM.test_special_values_hand_worked]),
    "overflow_via_carry": ("algorithm2", "if (e >= all_ones) return (s << 31) | 0x7F800000u;", "",
                           [T_AMSIM.test_special_values_hand_worked]),
    "mitchell_branch": ("orc_approx_mul", "(x + y < 1.0)", "(x + y < 2.0)",
                        [lambda o: T_AMSIM.test_mitchell_lut_is_log_domain_construction(o, 3)]),
    "mitchell_formula": ("orc_approx_mul", "(2.0 * (x + y))", "(x + y + 1.0)",
                         [T_AMSIM.test_mitchell_hand_values]),
    "exact_operand": ("orc_approx_mul", "p = (1.0 + x) * (1.0 + y);", "p = (1.0 + x) * (1.0 + x);",
                      [lambda o: T_AMSIM.test_exact_equals_ieee_product_all_mantissa_pairs(o, 5)]),
    "index_rounds": ("algorithm2", "uint32_t qa = top_bits(a, M), qb = top_bits(b, M);",
                     "uint32_t qa = top_bits(a + (1u << (22 - M)), M), qb = top_bits(b + (1u << (22 - M)), M);",
                     [lambda o: T_AMSIM.test_exact_equals_ieee_product_sampled(o, 9)]),
    "sign_dropped": ("algorithm2", "uint32_t s = sign_of(a) ^ sign_of(b);", "uint32_t s = sign_of(a);",
                     [T_AMSIM.test_mitchell_scaling_in_normal_range]),
    "denormal_not_zero": ("cast_operand", "if (ex == 0) return CL_ZERO;", "if (ex == 0) return CL_NORMAL;",
                          [T_AMSIM.test_zero_sign_and_denormals]),
    "gemm_transposed_a": ("orc_gemm_row", "g->ta ? g->A[(int64_t)kk * g->lda + i]",
                          "g->ta ? g->A[(int64_t)i * g->lda + kk]",
                          [lambda o: T_CONTR.test_gemm_exact_kind_equals_float64_matmul(o, True, False)]),
    "gemm_sumabs_signed": ("orc_gemm_row", "sa += fabs((double)p);", "sa += (double)p;",
                           [lambda o: T_CONTR.test_gemm_exact_kind_equals_float64_matmul(o, False, False)]),
    "conv_fwd_dilation_axis": ("orc_fwd_pt", "q * c->sw - c->pw + ss * c->dw, ch);", "q * c->sw - c->pw + ss * c->dh, ch);",
                               [lambda o: T_CONTR.test_conv_exact_kind_equals_torch_float64(o, T_CONTR.GEOMS[2])]),
    "conv_bwd_data_no_flip": ("orc_bwd_data_pt", "int hp = h + c->ph - r * c->dh", "int hp = h - c->ph + r * c->dh",
                              [lambda o: T_CONTR.test_conv_exact_kind_equals_torch_float64(o, T_CONTR.GEOMS[0])]),
    "conv_bwd_filter_pq_swap": ("orc_bwd_filter_pt", "(((int64_t)n * c->P + p) * c->Q + q)",
                                "(((int64_t)n * c->P + q) * c->Q + p)",
                                [lambda o: T_CONTR.test_conv_exact_kind_equals_torch_float64(o, T_CONTR.GEOMS[0])]),
    "dw_fwd_channel_split": ("orc_dw_fwd_pt", "int ch = k / D, d = k % D;", "int ch = k % c->C, d = k / c->C;",
                             [lambda o: T_CONTR.test_dwconv_exact_kind_equals_torch_grouped_float64(o, _dw_geom(1))]),
    "dw_bwd_data_channel": ("orc_dw_bwd_data_pt", "c->K + ch * D + d];", "c->K + d * c->C + ch];",
                            [lambda o: T_CONTR.test_dwconv_exact_kind_equals_torch_grouped_float64(o, _dw_geom(2))]),
    "dw_bwd_data_no_flip": ("orc_dw_bwd_data_pt", "int hp = h + c->ph - r * c->dh", "int hp = h - c->ph + r * c->dh",
                            [lambda o: T_CONTR.test_dwconv_exact_kind_equals_torch_grouped_float64(o, _dw_geom(0))]),
    "dw_bwd_filter_index_order": ("orc_dw_bwd_filter_pt", "int d = (int)(idx % D); idx /= D;\n    int ch = (int)(idx % c->C); idx /= c->C;",
                                  "int ch = (int)(idx % c->C); idx /= c->C;\n    int d = (int)(idx % D); idx /= D;",
                                  [lambda o: T_CONTR.test_dwconv_exact_kind_equals_torch_grouped_float64(o, _dw_geom(1))]),
    # user models (Algorithm 1 over a caller's approx_mul, Algorithm 2 over a stored table)
    "table_index_swapped": ("mult_entry", "mu->table[(qa << mu->M) | qb]", "mu->table[(qb << mu->M) | qa]",
                            [T_USER.test_asymmetric_model_hand_worked]),
    "table_carry_ignored": ("mult_entry", "*entry = mu->table[(qa << mu->M) | qb];",
                            "*entry = mu->table[(qa << mu->M) | qb] & 0x7FFFFFu;",
                            [T_USER.test_table_products_brute_force]),
    "user_carry_detection": ("algorithm1_entry", "else if (real_exp == un_normalized_exp + 1) carry = 1;",
                             "else if (real_exp == un_normalized_exp + 1) carry = 0;",
                             [lambda o: T_USER.test_exact_model_callback_gives_exact_kind(o, 4),
                              lambda o: T_AMSIM.test_exact_lut_is_integer_normalisation(o, 4)]),
    "user_negative_allowed": ("algorithm1_entry", "if (sign_of(uc)) return ORC_EINVAL;", "",
                              [T_USER.test_algorithm1_rejects_models_outside_its_range]),
    # (1, E, M) formats: the exponent cast and the re-biased Algorithm 2
    "cast_bias": ("cast_operand", "const int bias = (1 << (E - 1)) - 1;", "const int bias = (1 << (E - 1));",
                  [T_FMT.test_format_hand_worked]),
    "cast_underflow_boundary": ("cast_operand", "if (c <= 0) return CL_ZERO;", "if (c < 0) return CL_ZERO;",
                                [T_FMT.test_format_hand_worked]),
    "cast_overflow_boundary": ("cast_operand", "if (c >= all_ones) return CL_INF;", "if (c > all_ones) return CL_INF;",
                               [T_FMT.test_format_hand_worked]),
    "format_overflow_threshold": ("algorithm2", "const int all_ones = (1 << mu->E) - 1;",
                                  "const int all_ones = (1 << mu->E);",
                                  [lambda o: T_FMT.test_half_format_matches_ieee_half_ranges(o, "exact")]),
    "format_result_not_rebiased": ("algorithm2", "((uint32_t)(e - bias + 127) << 23)", "((uint32_t)e << 23)",
                                   [lambda o: T_FMT.test_half_format_matches_ieee_half_ranges(o, "exact")]),
}


def test_unmutated_oracle_passes_the_chosen_pins(tmp_path):
    o = _mutant_oracle(tmp_path, "algorithm2", "uint32_t s = sign_of(a) ^ sign_of(b);",
                       "uint32_t s = sign_of(a) ^ sign_of(b);")
    for _, _, _, pins in MUTANTS.values():
        for pin in pins:
            pin(o)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(tmp_path, name):
    fname, old, new, pins = MUTANTS[name]
    o = _mutant_oracle(tmp_path, fname, old, new)
    failed = 0
    for pin in pins:
        try:
            pin(o)
        except (AssertionError, ValueError, pytest.fail.Exception):
            failed += 1
    assert failed > 0, f"no pin caught the planted mistake {name}"
