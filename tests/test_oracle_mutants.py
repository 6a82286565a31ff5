"""Planted mistakes in copies of the oracle must each fail at least one pin.

Every mutant is a one-spot textual change to ``oracle/ssm_oracle.c`` of the
kind a careless rewrite makes (a dropped term, a wrong sign, a wrong index, a
transposed operand, an update out of order).  The copy is compiled into a
temporary library on the CPU; the real oracle is never touched.
"""

import os

import pytest

import pins
from oracle import oracle as orc

MUTANTS = {
    "drop_skip_term": ("double out = s + skip * u_c[t];", "double out = s;"),
    "exp_sign": ("const double abar = exp(dt * A_d[n]);", "const double abar = exp(-dt * A_d[n]);"),
    "read_before_update": (
        "h[n] = abar * h[n] + bbar * u_c[t];\n                s += C_b[n * seqlen + t] * h[n];",
        "s += C_b[n * seqlen + t] * h[n];\n                h[n] = abar * h[n] + bbar * u_c[t];"),
    "B_transposed": ("oracle_bbar(dt, A_d[n], B_b[n * seqlen + t], zoh)",
                     "oracle_bbar(dt, A_d[n], B_b[t * dstate + n], zoh)"),
    "B_C_swapped": ("s += C_b[n * seqlen + t] * h[n];", "s += B_b[n * seqlen + t] * h[n];"),
    "softplus_drops_x": ("return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));",
                         "return x > 0.0 ? log1p(exp(-x)) : log1p(exp(x));"),
    "bias_not_added": ("double dt = dt_c[t] + bias_d;", "double dt = dt_c[t];"),
    "first_order_drops_delta": ("return delta * b;\n    return expm1", "return b;\n    return expm1"),
    "zoh_missing_division": ("return expm1(delta * a) / a * b;", "return expm1(delta * a) * b;"),
    "gate_is_sigmoid": ("return x / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(-x));"),
    "h0_ignored": ("h[n] = h0 ? h0[c * dstate + n] : 0.0;", "h[n] = 0.0;"),
    "A_row_of_channel_0": ("const double *A_d = A + d * dstate;", "const double *A_d = A;"),
    "skip_of_channel_0": ("const double *A_d = A + d * dstate;\n        const double skip = Dskip ? Dskip[d] : 0.0;",
                          "const double *A_d = A + d * dstate;\n        const double skip = Dskip ? Dskip[0] : 0.0;"),
    "B_of_batch_0": ("const double *B_b = B + b * dstate * seqlen;", "const double *B_b = B;"),
    "gate_only_on_state_term": (
        "double out = s + skip * u_c[t];\n            if (z_c)\n                out *= oracle_silu(z_c[t]);",
        "double out = s;\n            if (z_c)\n                out *= oracle_silu(z_c[t]);\n            out += skip * u_c[t];"),
    "step_state_not_decayed": ("*h = abar * *h + bbar * u[c];", "*h = *h + bbar * u[c];"),
    "step_B_of_batch_0": ("oracle_bbar(dt, a, B[b * dstate + n], zoh)", "oracle_bbar(dt, a, B[n], zoh)"),
    "step_no_bias": ("double dt = delta[c] + (bias ? bias[d] : 0.0);", "double dt = delta[c];"),
    "conv_taps_reversed": ("acc += w[d * width + k] * ORACLE_X_AT(s);",
                           "acc += w[d * width + (width - 1 - k)] * ORACLE_X_AT(s);"),
    "conv_no_bias": ("double acc = bias ? bias[d] : 0.0;\n            for (int64_t k = 0; k < width; ++k) {",
                     "double acc = 0.0;\n            for (int64_t k = 0; k < width; ++k) {"),
    "conv_state_ignored": ("(s_c ? s_c[hist + (s)] : 0.0)", "0.0"),
    "conv_state_newest_first": ("(s_c ? s_c[hist + (s)] : 0.0)", "(s_c ? s_c[-(s) - 1] : 0.0)"),
    "conv_state_out_window": ("const int64_t s = seqlen - hist + j;", "const int64_t s = seqlen - width + j;"),
    "conv_no_silu": ("u[c * seqlen + t] = silu ? oracle_silu(acc) : acc;", "u[c * seqlen + t] = acc;"),
    "conv_step_no_shift": ("s_c[k] = s_c[k + 1];", "s_c[k] = s_c[k];"),
    "conv_step_current_tap": ("acc += w[d * width + hist] * x[c];", "acc += w[d * width] * x[c];"),
    "conv_step_taps_shifted": ("acc += w[d * width + k] * s_c[k];", "acc += w[d * width + k + 1] * s_c[k];"),
    "bwd_readout_not_in_lambda": ("lam[n] += C_b[n * L + t] * yhat;", "lam[n] += 0.0;"),
    "bwd_dA_missing_delta": ("dA[d * N + n] += dabar * abar * dt[t];", "dA[d * N + n] += dabar * abar;"),
    "bwd_ddt_missing_A": ("ddt += dabar * abar * a;", "ddt += dabar * abar;"),
    "bwd_softplus_grad_dropped": ("dx *= 1.0 / (1.0 + exp(-(dr_c[t] + bias_d)));", "dx *= 1.0;"),
    "bwd_dz_missing_silu_prime": ("dy_c[t] * pre[t] * sg * (1.0 + z_c[t] * (1.0 - sg));",
                                  "dy_c[t] * pre[t] * sg;"),
    "bwd_dC_uses_prev_state": ("dC[b * N * L + n * L + t] += yhat * h[(t + 1) * N + n];",
                               "dC[b * N * L + n * L + t] += yhat * h[t * N + n];"),
    "bwd_zoh_dB_first_order": ("dB[b * N * L + n * L + t] += dbbar * expm1(dt[t] * a) / a;",
                               "dB[b * N * L + n * L + t] += dbbar * dt[t];"),
    "bwd_no_decay_propagation": ("lam[n] *= abar;", "lam[n] *= 1.0;"),
    "bwd_dD_missing": ("dDskip[d] += yhat * u_c[t];", "dDskip[d] += 0.0;"),
    "ssd_no_decay": ("S[p * N + n] = a * S[p * N + n] + d * Bt[n] * xt[p];",
                     "S[p * N + n] = S[p * N + n] + d * Bt[n] * xt[p];"),
    "ssd_input_without_delta": ("S[p * N + n] = a * S[p * N + n] + d * Bt[n] * xt[p];",
                                "S[p * N + n] = a * S[p * N + n] + Bt[n] * xt[p];"),
    "ssd_readout_with_B": ("acc += S[p * N + n] * Ct[n];", "acc += S[p * N + n] * Bt[n];"),
    "ssd_skip_dropped": ("yt[p] = acc + (Dskip ? Dskip[h] : 0.0) * xt[p];", "yt[p] = acc;"),
    "ssd_dt_bias_dropped": ("double d = dt[(b * L + t) * H + h] + (dt_bias ? dt_bias[h] : 0.0);",
                            "double d = dt[(b * L + t) * H + h];"),
    "ssd_A_of_head_0": ("const double a = exp(d * A[h]);", "const double a = exp(d * A[0]);"),
    # mistakes that break linearity in the input (caught by superposition, P16)
    "state_update_constant_term": ("h[n] = abar * h[n] + bbar * u_c[t];",
                                   "h[n] = abar * h[n] + bbar * u_c[t] + 1e-3 * dt;"),
    "skip_term_squared": ("double out = s + skip * u_c[t];", "double out = s + skip * u_c[t] * fabs(u_c[t]);"),
}


@pytest.fixture(scope="module")
def source():
    with open(orc.source_path()) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutant {name}: anchor not found exactly once"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    so = orc.build(str(src), str(tmp_path / f"lib{name}.so"), force=True)
    lib = orc.load(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"


def test_unmutated_copy_passes(source, tmp_path):
    src = tmp_path / "same.c"
    src.write_text(source)
    lib = orc.load(orc.build(str(src), str(tmp_path / "libsame.so"), force=True))
    for pin in pins.ALL_PINS:
        pin(lib)
    assert os.path.exists(str(tmp_path / "libsame.so"))
