"""Plant a plausible mistake in a copy of the oracle's C source, build it, and
check that at least one pin fails.  This shows the pins constrain every part
of the oracle: a dropped term, a wrong sign, divisor or index, a swapped
operand.  CPU only; the committed oracle is never modified."""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "norm_oracle.c")

MUTATIONS = {
    "ln_unbiased_variance": ("double var = ssd / (double)cols;",
                             "double var = ssd / (double)(cols - 1);"),
    "ln_eps_outside_root": ("double rs = 1.0 / sqrt(var + eps);",
                            "double rs = 1.0 / (sqrt(var) + eps);"),
    "ln_bwd_eps_outside_root": ("double rs = 1.0 / sqrt(ssd / (double)cols + eps);",
                                "double rs = 1.0 / (sqrt(ssd / (double)cols) + eps);"),
    "ln_bwd_unbiased_variance": ("double rs = 1.0 / sqrt(ssd / (double)cols + eps);",
                                 "double rs = 1.0 / sqrt(ssd / (double)(cols - 1) + eps);"),
    "rms_fwd_eps_outside_root": (
        "double rr = 1.0 / sqrt(ss / (double)cols + eps);\n        for (int64_t j = 0; j < cols; ++j)\n            y[",
        "double rr = 1.0 / (sqrt(ss / (double)cols) + eps);\n        for (int64_t j = 0; j < cols; ++j)\n            y["),
    "rms_bwd_eps_outside_root": ("double rr = 1.0 / sqrt(ss / (double)cols + eps);\n\n        double s = 0.0;",
                                 "double rr = 1.0 / (sqrt(ss / (double)cols) + eps);\n\n        double s = 0.0;"),
    "bn_fwd_eps_outside_root": ("rs = 1.0 / sqrt(var_biased + eps);", "rs = 1.0 / (sqrt(var_biased) + eps);"),
    "bn_bwd_eps_outside_root": ("rs = 1.0 / sqrt(ssd / (double)m + eps);",
                                "rs = 1.0 / (sqrt(ssd / (double)m) + eps);"),
    "bn_eval_fwd_drops_eps": ("rs = 1.0 / sqrt(running_var[ch] + eps);\n        }\n        if (save_mean)",
                              "rs = 1.0 / sqrt(running_var[ch]);\n        }\n        if (save_mean)"),
    "ln_bwd_drops_xhat_term": ("- xhat * sum_gxhat / (double)cols);", ");"),
    "ln_bwd_mean_term_divisor": ("rs * (g - sum_g / (double)cols",
                                 "rs * (g - sum_g / (double)(cols - 1)"),
    "ln_dw_uses_x_not_xhat": ("if (dw) dw[j] += dyr[j] * xhat;",
                              "if (dw) dw[j] += dyr[j] * xr[j];"),
    "ln_db_sign": ("if (db) db[j] += dyr[j];", "if (db) db[j] -= dyr[j];"),
    "rms_fwd_drops_weight": ("y[r * cols + j] = xr[j] * rr * (w ? w[j] : 1.0) + (b ? b[j] : 0.0);",
                             "y[r * cols + j] = xr[j] * rr + (b ? b[j] : 0.0);"),
    "rms_fwd_drops_bias": ("y[r * cols + j] = xr[j] * rr * (w ? w[j] : 1.0) + (b ? b[j] : 0.0);",
                           "y[r * cols + j] = xr[j] * rr * (w ? w[j] : 1.0);"),
    "rms_db_scaled_by_x": ("if (db) db[j] = db[j] + dyr[j];", "if (db) db[j] = db[j] + dyr[j] * xr[j];"),
    "rms_bwd_rstd_squared": ("xr[j] * rr * rr * rr * s", "xr[j] * rr * rr * s"),
    "rms_bwd_term_sign": ("dx[r * cols + j] = rr * g - xr[j]",
                          "dx[r * cols + j] = rr * g + xr[j]"),
    "bn_normalise_unbiased": ("double var_biased = ssd / (double)m;",
                              "double var_biased = ssd / (double)(m - 1);"),
    "bn_running_var_biased": ("momentum * var_unbiased", "momentum * var_biased"),
    "bn_momentum_swapped": ("(1.0 - momentum) * running_mean[ch] + momentum * mu",
                            "momentum * running_mean[ch] + (1.0 - momentum) * mu"),
    "bn_residual_after_activation": (
        "y[e] = act_forward(act, act_param, z);",
        "y[e] = act_forward(act, act_param, z - (res ? res[e] : 0.0)) + (res ? res[e] : 0.0);"),
    "leaky_relu_slope_on_positive_side": ("case ORACLE_ACT_LEAKY_RELU: return z > 0.0 ? z : param * z;",
                                          "case ORACLE_ACT_LEAKY_RELU: return z > 0.0 ? param * z : z;"),
    "leaky_relu_grad_ignores_slope": ("case ORACLE_ACT_LEAKY_RELU: return z > 0.0 ? 1.0 : param;",
                                      "case ORACLE_ACT_LEAKY_RELU: return z > 0.0 ? 1.0 : 0.0;"),
    "elu_without_minus_one": ("case ORACLE_ACT_ELU: return z > 0.0 ? z : param * expm1(z);",
                              "case ORACLE_ACT_ELU: return z > 0.0 ? z : param * exp(z);"),
    "sigmoid_grad_missing_one_minus": ("        return s * (1.0 - s);\n    }\n    case ORACLE_ACT_CELU",
                                       "        return s;\n    }\n    case ORACLE_ACT_CELU"),
    "celu_without_scaled_exponent": ("case ORACLE_ACT_CELU: return z > 0.0 ? z : param * expm1(z / param);",
                                     "case ORACLE_ACT_CELU: return z > 0.0 ? z : param * expm1(z);"),
    "selu_positive_side_unscaled": ("case ORACLE_ACT_SELU: return z > 0.0 ? SELU_LAMBDA * z :",
                                    "case ORACLE_ACT_SELU: return z > 0.0 ? z :"),
    "elu_grad_drops_exp": ("case ORACLE_ACT_ELU: return z > 0.0 ? 1.0 : param * exp(z);",
                           "case ORACLE_ACT_ELU: return z > 0.0 ? 1.0 : param;"),
    "bn_gelu_grad_drops_pdf_term": ("return cdf + z * pdf;", "return cdf;"),
    "relu6_no_upper_clamp": ("case ORACLE_ACT_RELU6: return z < 0.0 ? 0.0 : (z > 6.0 ? 6.0 : z);",
                             "case ORACLE_ACT_RELU6: return z < 0.0 ? 0.0 : z;"),
    "relu6_grad_at_upper_end": ("case ORACLE_ACT_RELU6: return (z > 0.0 && z < 6.0) ? 1.0 : 0.0;",
                                "case ORACLE_ACT_RELU6: return (z > 0.0 && z <= 6.0) ? 1.0 : 0.0;"),
    "hardtanh_lower_bound_zero": ("case ORACLE_ACT_HARDTANH: return z < -1.0 ? -1.0 : (z > 1.0 ? 1.0 : z);",
                                  "case ORACLE_ACT_HARDTANH: return z < 0.0 ? 0.0 : (z > 1.0 ? 1.0 : z);"),
    "hardtanh_grad_ignores_range": ("case ORACLE_ACT_HARDTANH: return (z > -1.0 && z < 1.0) ? 1.0 : 0.0;",
                                    "case ORACLE_ACT_HARDTANH: return 1.0;"),
    "bn_relu_grad_at_zero": ("case ORACLE_ACT_RELU: return z > 0.0 ? 1.0 : 0.0;",
                             "case ORACLE_ACT_RELU: return z >= 0.0 ? 1.0 : 0.0;"),
    "bn_mask_bit_order": ("|= (uint32_t)1u << (j % 32);", "|= (uint32_t)1u << (31 - j % 32);"),
    "bn_dx_drops_mean_term": ("(dz - sum_dz / (double)m - xhat", "(dz - xhat"),
    "bn_dw_not_xhat": ("sum_dz_xhat += dz * xhat;", "sum_dz_xhat += dz * x[e];"),
    "bn_eval_dx_drops_weight": ("dx[e] = wc * rs * dz;", "dx[e] = rs * dz;"),
    "ln_cf_divides_by_positions": ("double var = ssd / (double)c;", "double var = ssd / (double)l;"),
    "ln_cf_dw_uses_x": ("if (dw) dw[ch] += dy[base + ch * l] * xhat;",
                        "if (dw) dw[ch] += dy[base + ch * l] * x[base + ch * l];"),
    "silu_uses_tanh": ("case ORACLE_ACT_SILU: return z * sigmoid(z);",
                       "case ORACLE_ACT_SILU: return z * tanh(z);"),
    "silu_grad_drops_product_term": ("return s + z * s * (1.0 - s);", "return s;"),
    "mish_softplus_without_log": ("case ORACLE_ACT_MISH: return z * tanh(softplus(z));",
                                  "case ORACLE_ACT_MISH: return z * tanh(exp(z));"),
    "mish_grad_wrong_chain_factor": ("return t + z * (1.0 - t * t) * sigmoid(z);",
                                     "return t + z * (1.0 - t * t);"),
    "philox_no_key_schedule": ("        k0 += 0x9E3779B9u;\n", ""),
    "philox_hi_lo_swapped": ("uint32_t n1 = (uint32_t)p1;", "uint32_t n1 = (uint32_t)(p1 >> 32);"),
    "dropout_scale_not_inverted": ("? a / (1.0 - drop_p) : 0.0;", "? a * (1.0 - drop_p) : 0.0;"),
    "dropout_window_ignores_first": ("y[i] = dropout_keep(seed, first + i, drop_p)", "y[i] = dropout_keep(seed, i, drop_p)"),
    "dropout_keep_flipped": ("return !(u < (float)drop_p);", "return u < (float)drop_p;"),
    "dropout_one_word_per_call": ("out[e & 3] >> 8", "out[0] >> 8"),
    "dropout_bwd_drops_scale": ("dx[i] = dy[i] / (1.0 - drop_p) * act_derivative(act, act_param, x[i]);",
                                "dx[i] = dy[i] * act_derivative(act, act_param, x[i]);"),
    "dropout_bwd_mask_ignored": ("        if (dropout_keep(seed, first + i, drop_p))\n            dx[i]",
                                 "        if (1)\n            dx[i]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor must occur once: {old!r}"
    mutated = tmp_path / "norm_oracle.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(src=str(mutated), out=str(tmp_path / "libmutant.so"), force=True)
    o = oracle.Oracle(lib)
    for pin in PINS:
        try:
            pin(o)
        except AssertionError:
            return
        except FloatingPointError:
            return
    pytest.fail(f"no pin caught the planted mistake {name}")
