"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch each one: a wrong bias or fraction width, a dropped term, a
wrong sign, a wrong tie rule, a swapped operand or lane, a wrong clamp.

Each mutant is oracle.c with one textual substitution, compiled with the same
flags into a temporary directory and loaded through oracle.Oracle; the listed
pins must raise AssertionError on it.
"""
import os

import pytest

import oracle
import pins

with open(oracle.SOURCE) as _f:
    _SRC = _f.read()

# (name, original text, planted text, pins expected to fail -- at least one must)
MUTANTS = [
    ("bias_14", "#define E4_BIAS 15", "#define E4_BIAS 14",
     ["e4_closed_forms", "e4_shared_binary16_codes"]),
    ("e4m11_fraction_10_bits",
     "e4m11_mag[c] = (float)ieee_style_value(c >> 11, c & 0x7FFu, 11, E4_BIAS);",
     "e4m11_mag[c] = (float)ieee_style_value(c >> 11, c & 0x7FFu, 10, E4_BIAS);",
     ["e4_equal_spacing_and_sign", "e4_closed_forms"]),
    ("subnormal_exponent_off_by_one",
     "return ldexp((double)f, 1 - bias - mbits);",
     "return ldexp((double)f, - bias - mbits);",
     ["e4_shared_binary16_codes", "e4_closed_forms"]),
    ("ties_to_odd", "return (lo % 2u == 0u) ? lo : hi;", "return (lo % 2u == 0u) ? hi : lo;",
     ["e4_encode_textbook_rne", "e4_encode_brute_force"]),
    ("ties_away", "return (lo % 2u == 0u) ? lo : hi;", "return hi;",
     ["e4_encode_textbook_rne"]),
    ("no_saturation", "if (ax >= t[count - 1])\n        return count - 1;",
     "if (ax >= t[count - 1])\n        return 0;",
     ["e4_specials", "e4_encode_textbook_rne"]),
    ("negative_zero_lost",
     "return (uint16_t)((signbit(x) ? 0x8000u : 0u) | mag);\n}\n\n/* ---- E4M12",
     "return (uint16_t)((x < 0.0f ? 0x8000u : 0u) | mag);\n}\n\n/* ---- E4M12",
     ["e4_roundtrip_all_codes", "e4_specials"]),
    ("weight_decay_dropped", "h.dk = (float)(1.0 - lr * wd);", "h.dk = 1.0f;",
     ["step1_closed_form_e4", "fp32_matches_torch_adamw", "zero_gradient_decay_fp32"]),
    ("weight_decay_coupled_sign", "h.dk = (float)(1.0 - lr * wd);", "h.dk = (float)(1.0 + lr * wd);",
     ["step1_closed_form_e4", "fp32_matches_torch_adamw"]),
    ("bias_correction1_dropped",
     "h.ss = (float)(lr / (1.0 - pow(beta1, (double)step)));", "h.ss = (float)lr;",
     ["step1_closed_form_e4", "fp32_matches_torch_adamw"]),
    ("bias_correction2_dropped",
     "h.bc2 = (float)(1.0 - pow(beta2, (double)step));", "h.bc2 = 1.0f;",
     ["step1_closed_form_e4", "fp32_matches_torch_adamw"]),
    ("update_sign", "*p_new = pd - upd;", "*p_new = pd + upd;",
     ["step1_closed_form_fp32"]),
    ("gradient_not_squared", "float t2 = t * g;", "float t2 = t;",
     ["step1_closed_form_fp32", "fp32_matches_torch_adamw"]),
    ("beta1_in_second_moment", "float v1 = h->b2 * v;", "float v1 = h->b1 * v;",
     ["fp32_matches_torch_adamw"]),
    ("eps_dropped", "float den = s + h->ef;", "float den = s;",
     ["step1_closed_form_fp32", "fp32_matches_torch_adamw"]),
    ("first_moment_no_decay", "float m1 = h->b1 * m;", "float m1 = m;",
     ["fp32_matches_torch_adamw"]),
    ("rms_not_squared", "float v = r * r;", "float v = r;",
     ["packed_e4_is_fp32_on_decoded"]),
    ("stores_v_not_rms", "float rn = sqrtf(vn);", "float rn = vn;",
     ["step1_closed_form_e4", "packed_e4_is_fp32_on_decoded"]),
    ("stores_corrected_rms", "float rn = sqrtf(vn);", "float rn = sqrtf(vn / h.bc2);",
     ["step1_closed_form_e4", "packed_e4_is_fp32_on_decoded"]),
    ("lanes_swapped",
     "state[i] = ((uint32_t)oracle_e4m12_encode(rn) << 16) | oracle_e4m11_encode(mn);",
     "state[i] = ((uint32_t)oracle_e4m11_encode(mn) << 16) | oracle_e4m12_encode(rn);",
     ["step1_closed_form_e4", "packed_e4_is_fp32_on_decoded"]),
    ("fp16_no_saturation", "uint32_t mag = nearest_code(fp16_mag, 31u << 10, fabsf(x));",
     "uint32_t mag = fabsf(x) >= 65520.0f ? 0x7C00u : nearest_code(fp16_mag, 31u << 10, fabsf(x));",
     ["fp16_specials"]),
    ("midpoint_tie_upward", "if (mid[j] < c)", "if (mid[j] <= c)",
     ["requantise_matches_torch_spec", "requantise_searchsorted"]),
    ("absmax_floor_wrong", "#define ABSMAX_FLOOR 1e-30f", "#define ABSMAX_FLOOR 1e-20f",
     ["requantise_matches_torch_spec", "requantise_searchsorted"]),
    ("absmax_stored_clamped", "*absmax_out = a;", "*absmax_out = scale;",
     ["requantise_brute_force_and_invariants", "requantise_searchsorted"]),
    ("absmax_signed_max", "float ax = fabsf(x[i]);", "float ax = x[i];",
     ["requantise_matches_torch_spec", "requantise_searchsorted"]),
    ("midpoint_not_halved", "mid[j] = s * 0.5f;", "mid[j] = s * 0.25f;",
     ["requantise_matches_torch_spec", "requantise_searchsorted"]),
    ("dequantise_wrong_map", "float v = qmap2[v_code[i]] * av;", "float v = qmap1[v_code[i]] * av;",
     ["blockwise_step_composition"]),
    ("bf16_truncates", "pick = (lo % 2u == 0u) ? lo : lo + 1u;", "pick = lo;",
     ["bf16_matches_torch"]),
    # re-associations and contractions: the same algebra, other roundings
    ("gradient_squared_first", "float t = h->c2 * g;\n    float t2 = t * g;",
     "float t = g * g;\n    float t2 = h->c2 * t;", ["fp32_element_matches_page_spec"]),
    ("step_size_after_division", "float u = h->ss * mn;\n    float upd = u / den;",
     "float u = mn / den;\n    float upd = h->ss * u;", ["fp32_element_matches_page_spec"]),
    ("root_of_each_factor", "float q = vn / h->bc2;\n    float s = sqrtf(q);",
     "float q = sqrtf(vn);\n    float s = q / sqrtf(h->bc2);", ["fp32_element_matches_page_spec"]),
    ("bc2_by_reciprocal", "float q = vn / h->bc2;", "float q = vn * (1.0f / h->bc2);",
     ["fp32_element_matches_page_spec"]),
    ("first_moment_contracted", "float mn = m1 + m2;", "float mn = fmaf(h->b1, m, m2);",
     ["fp32_element_matches_page_spec"]),
    ("decay_line_contracted", "*p_new = pd - upd;", "*p_new = fmaf(p, h->dk, -upd);",
     ["fp32_element_matches_page_spec"]),
    ("decay_after_update", "float pd = p * h->dk;\n    *p_new = pd - upd;",
     "float pd = p - upd;\n    *p_new = pd * h->dk;", ["fp32_element_matches_page_spec"]),
    ("one_minus_beta_in_float", "h.c1 = (float)(1.0 - beta1);", "h.c1 = 1.0f - (float)beta1;",
     ["fp32_element_matches_page_spec"]),
]


@pytest.mark.parametrize("name,old,new,expect", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, expect, tmp_path):
    assert _SRC.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = tmp_path / f"{name}.c"
    src.write_text(_SRC.replace(old, new, 1))
    lib = oracle.compile_source(str(src), str(tmp_path / f"{name}.so"))
    orc = oracle.Oracle(os.path.abspath(lib))
    caught = []
    for pin in expect:
        try:
            pins.ALL_CHECKS[pin](orc)
        except AssertionError:
            caught.append(pin)
    assert caught, f"planted mistake {name} passed every pin in {expect}"
