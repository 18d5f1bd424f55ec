"""Plants plausible mistakes in copies of the oracle (on the CPU) and checks
that the pins catch every one: a dropped term, a wrong sign, a wrong index, a
transposed operand, a wrong reading of the variance or of eps."""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "ln_eps_dropped": ("*r = 1.0 / sqrt(v + eps);", "*r = 1.0 / sqrt(v);"),
    "ln_unbiased_var": ("double v = q / (double)n;", "double v = q / (double)(n - 1);"),
    "ln_uncentred_var": ("q += (x[j] - m) * (x[j] - m);", "q += x[j] * x[j];"),
    "rms_eps_outside_root": ("*r = 1.0 / sqrt(ms + eps);", "*r = 1.0 / (sqrt(ms) + eps);"),
    "rms_mean_not_sum": ("double ms = q / (double)n;", "double ms = q;"),
    "weight_one_plus_gamma": ("y[j] = xhat * gamma[j] + b;", "y[j] = xhat * (1.0 + gamma[j]) + b;"),
    "beta_dropped": ("y[j] = xhat * gamma[j] + b;", "y[j] = xhat * gamma[j];"),
    "fwd_mean_not_subtracted": ("double xhat = (x[j] - mu) * r;\n        double b",
                                "double xhat = x[j] * r;\n        double b"),
    "dx_sign": ("dx[j] = r * (g - a - xhat * c);", "dx[j] = r * (g - a + xhat * c);"),
    "dx_rstd_dropped": ("dx[j] = r * (g - a - xhat * c);", "dx[j] = (g - a - xhat * c);"),
    "dx_mean_g_dropped": ("double a = (mode == ORACLE_LAYER) ? sum_g / (double)n : 0.0;",
                          "double a = 0.0;"),
    "c_missing_gamma": ("sum_gxhat += g * xhat;", "sum_gxhat += dy[j] * xhat;"),
    "c_not_mean": ("double c = sum_gxhat / (double)n;", "double c = sum_gxhat;"),
    "dgamma_x_not_xhat": ("dgamma[j] += dy[j] * xhat;", "dgamma[j] += dy[j] * x[j];"),
    "dbeta_times_gamma": ("dbeta[j] += dy[j];", "dbeta[j] += dy[j] * gamma[j];"),
    "widen_wrong_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "row_index_k": ("widen_row(x + i * N, N, xr);\n        double mu, r;",
                    "widen_row(x + k * N, N, xr);\n        double mu, r;"),
    "param_grads_transposed": ("widen_row(x + i * N, N, xr);\n        widen_row(dy + i * N, N, dyr);\n        bwd_row(dyr, xr, g, N, eps, mode, NULL",
                               "widen_row(x + i * N, N, xr);\n        widen_row(dy + i * N, N, dyr);\n        bwd_row(xr, dyr, g, N, eps, mode, NULL"),
    "residual_round_truncates": ("u += 0x7FFFu + lsb;", "u += 0u * lsb;"),
    "residual_ties_away": ("u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;"),
    "residual_dh_subtracted": ("dx[k * N + j] += bf16_bits_to_double(dh[i * N + j]);",
                               "dx[k * N + j] -= bf16_bits_to_double(dh[i * N + j]);"),
    "residual_dh_wrong_row": ("dx[k * N + j] += bf16_bits_to_double(dh[i * N + j]);",
                              "dx[k * N + j] += bf16_bits_to_double(dh[k * N + j]);"),
    "e4m3_round_toward_zero": ("double m = nearbyint(ldexp(a, 3 - e));",
                               "double m = trunc(ldexp(a, 3 - e));"),
    "e4m3_subnormal_spacing": ("double m = nearbyint(ldexp(a, 9));",
                               "double m = nearbyint(ldexp(a, 8));"),
    "e4m3_decode_bias": ("v = ldexp((double)(8 + m), e - 10);",
                         "v = ldexp((double)(8 + m), e - 11);"),
    "e4m3_overflow_to_nan": ("if (a >= E4M3_MAX)\n        return sign | 0x7E;",
                             "if (a >= E4M3_MAX)\n        return sign | 0x7F;"),
    "fp8_row_max_240": ("e4m3_code(am > 0.0 ? (yk[j] / am) * E4M3_MAX : yk[j]);",
                        "e4m3_code(am > 0.0 ? (yk[j] / am) * 240.0 : yk[j]);"),
    "fp8_row_scale_inverted": ("scale[k] = am > 0.0 ? am / E4M3_MAX : 1.0;",
                               "scale[k] = am > 0.0 ? E4M3_MAX / am : 1.0;"),
    "mx_emax_7": ("e = (e2 - 1) - 8;", "e = (e2 - 1) - 7;"),
    "mx_no_clamp": ("if (e < -127)\n                        e = -127;",
                    "if (e < -227)\n                        e = -127;"),
    "mx_scale_applied_inverted": ("e4m3_code(ldexp(yb[j], -e));", "e4m3_code(ldexp(yb[j], e));"),
    "mx_amax_half_block": ("for (int j = 0; j < MX_BLOCK; ++j)\n                    if (fabs(yb[j]) > am)",
                           "for (int j = 0; j < MX_BLOCK / 2; ++j)\n                    if (fabs(yb[j]) > am)"),
    "gemm_w_transposed": ("s += yr[j] * wr[j];",
                          "s += yr[j] * bf16_bits_to_double(w[j * Nout + o]);"),
    "gemm_x_not_y": ("s += yr[j] * wr[j];", "s += xr[j] * wr[j];"),
    "gemm_one_w_row": ("widen_row(w + o * K, K, wr);", "widen_row(w, K, wr);"),
    "gemm_gamma_twice": ("s += yr[j] * wr[j];", "s += yr[j] * wr[j] * g[j];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    cfile = tmp_path / "mutant.c"
    cfile.write_text(mutated)
    lib = oracle.compile_c(str(cfile), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, FloatingPointError, ValueError, RuntimeError) as e:
            caught.append((pin.__name__, str(e)[:80]))
            break
    assert caught, f"mutant {name} passed every pin"
