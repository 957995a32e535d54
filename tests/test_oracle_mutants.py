"""Planted mistakes in a copy of the oracle must each break at least one pin.

Every entry edits one plausible spot of the oracle's C source (a dropped term,
a wrong sign, exponent or index, a wrong rounding rule), compiles the edited
copy on the CPU and runs all pins against it.  A mutant that passes every pin
would mean the pins cannot tell that mistake from the oracle.
"""
import os

import pytest

import oracle
import oracle_pins

# (name, text to replace, replacement, which occurrence)
MUTANTS = [
    ("eps_added_to_sum", "ss / (double)H + eps", "(ss + eps) / (double)H", 0),
    ("mean_over_H_minus_1", "ss / (double)H + eps", "ss / (double)(H + 1) + eps", 0),
    ("rstd_not_inverted", "double rstd = 1.0 / sqrt(", "double rstd = 1.0 * sqrt(", 0),
    ("bias_dropped", "(float)(wj + (double)weight_bias)", "(float)(wj)", 0),
    ("dx_sign", "rstd * g[j] * w_eff[j] - h[j] * r3 * m", "rstd * g[j] * w_eff[j] + h[j] * r3 * m", 0),
    ("dx_r_squared", "double r3 = rstd * rstd * rstd;", "double r3 = rstd * rstd;", 0),
    ("dx_m_no_weight", "dot += g[j] * w_eff[j] * h[j];", "dot += g[j] * h[j];", 0),
    ("dx_m_not_mean", "double m = dot / (double)H;", "double m = dot;", 0),
    ("dw_no_rstd", "dw_row[j] = g[j] * h[j] * rstd;", "dw_row[j] = g[j] * h[j];", 0),
    ("g_res_subtracted", "d += g_res[j];", "d -= g_res[j];", 0),
    ("bf16_ties_away", "double k = rint(ldexp(a, 7 - E));", "double k = round(ldexp(a, 7 - E));", 0),
    ("bf16_truncates", "double k = rint(ldexp(a, 7 - E));", "double k = floor(ldexp(a, 7 - E));", 0),
    ("bf16_decode_bias", "v = ldexp((double)(128 + f), e - 127 - 7);", "v = ldexp((double)(128 + f), e - 128 - 7);", 0),
    ("e4m3_decode_bias", "v = ldexp((double)(8 + f), e - 7 - 3);", "v = ldexp((double)(8 + f), e - 8 - 3);", 0),
    ("e4m3_ties_away", "double k = rint(ldexp(a, 3 - E));", "double k = round(ldexp(a, 3 - E));", 0),
    ("e4m3_no_saturation", "        return sign | 0x7E;", "        return sign | 0x7F;", 0),
    ("e5m2_decode_bias", "v = ldexp((double)(4 + f), e - 15 - 2);", "v = ldexp((double)(4 + f), e - 16 - 2);", 0),
    ("residual_not_rounded", "h[j] = orc_bf16_to_f64(hn);", "h[j] = xj + uj;", 0),
    ("quant_multiplies_scale", "double v = yv[j] / (double)scale;", "double v = yv[j] * (double)scale;", 0),
    ("block_scale_240", "float s = (float)(amax / 448.0);", "float s = (float)(amax / 240.0);", 0),
    ("block_scale_transposed", "block_scale[b * ldT + t] = s;", "block_scale[t * (H / 128) + b] = s;", 0),
    ("ada_no_one_plus", "double ov = yv[j] * (1.0 + sc) + sh;", "double ov = yv[j] * sc + sh;", 0),
    ("ada_shift_dropped", "double ov = yv[j] * (1.0 + sc) + sh;", "double ov = yv[j] * (1.0 + sc);", 0),
    ("ada_gate_from_shift", "gate_out[t * D + j] = st[2 * D + j];", "gate_out[t * D + j] = st[D + j];", 0),
    ("ada_style_row_zero", "(style_rows == 1 ? 0 : t)", "(style_rows == 1 ? 0 : 0)", 0),
    ("gated_product_unrounded", "double prod = orc_bf16_to_f64(orc_bf16_from_f64(xg));", "double prod = xg;", 0),
    ("gated_gate_from_shift", "gate_out[t * D + j] = st[2 * D + j];", "gate_out[t * D + j] = st[D + j];", 1),
    ("gated_no_one_plus", "double v = (yv[j] * (1.0 + sc) + sh) / (double)scale;", "double v = (yv[j] * sc + sh) / (double)scale;", 0),
    ("silu_exp_sign", "double s = yv[j] / (1.0 + exp(-yv[j]));", "double s = yv[j] / (1.0 + exp(yv[j]));", 0),
    ("silu_sigmoid_only", "double s = yv[j] / (1.0 + exp(-yv[j]));", "double s = 1.0 / (1.0 + exp(-yv[j]));", 0),
    ("silu_fp8_multiplies", "double v = s / (double)scale;", "double v = s * (double)scale;", 0),
    ("ln_unbiased_var", "double var = sq / (double)H;", "double var = sq / (double)(H - 1);", 0),
    ("ln_beta_dropped", "* rstd * (double)gamma[j] + (double)beta[j];", "* rstd * (double)gamma[j];", 0),
    ("ln_not_centred", "double o = (h[j] - mean) * rstd", "double o = h[j] * rstd", 0),
    ("ln_eps_outside_root", "1.0 / sqrt(var + (double)eps)", "1.0 / (sqrt(var) + (double)eps)", 0),
    ("ln_quant_formats_swapped", "fp8_kind ? orc_e5m2_from_f32(v32) : orc_e4m3_from_f32(v32)", "fp8_kind ? orc_e4m3_from_f32(v32) : orc_e5m2_from_f32(v32)", 1),
]


def _mutate(src, old, new, occ):
    pos = -1
    for _ in range(occ + 1):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    src = oracle.source_text()
    assert src.count(old) > occ, f"mutation site for {name} not found"
    path = oracle.compile_variant(_mutate(src, old, new, occ), os.path.join(tmp_path, f"{name}.so"))
    mutant = oracle.Oracle(oracle.load_path(path))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError) as e:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"


# Planted mistakes in the epilogues that a hand-derived golden alone must
# catch (not only the pins that compare the oracle with itself).
GOLDEN_CAUGHT = ["quant_multiplies_scale", "e4m3_no_saturation", "ada_no_one_plus",
                 "ada_shift_dropped", "ada_gate_from_shift", "gated_gate_from_shift",
                 "gated_no_one_plus", "silu_exp_sign", "silu_sigmoid_only", "silu_fp8_multiplies",
                 "ln_unbiased_var", "ln_beta_dropped", "ln_not_centred", "ln_eps_outside_root",
                 "ln_quant_formats_swapped", "block_scale_240", "dx_sign", "eps_added_to_sum"]


@pytest.mark.parametrize("name", GOLDEN_CAUGHT)
def test_golden_catches_mutant(tmp_path, name):
    old, new, occ = next((m[1], m[2], m[3]) for m in MUTANTS if m[0] == name)
    src = oracle.source_text()
    path = oracle.compile_variant(_mutate(src, old, new, occ), os.path.join(tmp_path, f"{name}.so"))
    mutant = oracle.Oracle(oracle.load_path(path))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        if not pin.__name__.startswith("pin_golden"):
            continue
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
            caught.append(pin.__name__)
    assert caught, f"no hand-derived golden catches the planted mistake {name}"
