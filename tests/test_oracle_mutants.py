"""Each plausible mistake planted in a copy of the oracle (on the CPU) must be
caught by at least one pin.  This shows the pins constrain every step."""
import os

import pytest

import oracle
from oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "scan_oracle.c")

# (name, text in scan_oracle.c, replacement)
MUTANTS = [
    ("output_reads_state_before_update",
     "h[n] = abar * h[n] + bbar_u;                /* state update       */\n"
     "            acc += Cb[t * N + n] * h[n];                /* C . state          */",
     "acc += Cb[t * N + n] * h[n];\n            h[n] = abar * h[n] + bbar_u;"),
    ("dropped_D_skip", "const double yt = acc + Dd * ut;", "const double yt = acc;"),
    ("sigmoid_gate_instead_of_silu", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("A_is_minus_A_log", "A[n] = -exp(j->A_log[d * N + n]);", "A[n] = -j->A_log[d * N + n];"),
    ("A_positive", "A[n] = -exp(j->A_log[d * N + n]);", "A[n] = exp(j->A_log[d * N + n]);"),
    ("Bbar_without_dt", "const double bbar_u = dt * Bb[t * N + n] * ut;",
     "const double bbar_u = Bb[t * N + n] * ut;"),
    ("Bbar_exact_zoh", "const double bbar_u = dt * Bb[t * N + n] * ut;",
     "const double bbar_u = (abar - 1.0) / A[n] * Bb[t * N + n] * ut;"),
    ("softplus_ignored", "j->softplus_flag ? oracle_softplus(raw) : raw", "raw"),
    ("softplus_positive_branch_wrong", "if (x > 0.0) return x + log1p(exp(-x));",
     "if (x > 0.0) return log1p(exp(-x));"),
    ("bias_ignored", "const double raw = dl[t] + bias;", "const double raw = dl[t];"),
    ("B_transposed", "const double bbar_u = dt * Bb[t * N + n] * ut;",
     "const double bbar_u = dt * Bb[n * L + t] * ut;"),
    ("C_is_B", "acc += Cb[t * N + n] * h[n];", "acc += Bb[t * N + n] * h[n];"),
    ("B_ignores_batch", "const double *Bb = j->B + b * L * N;", "const double *Bb = j->B;"),
    ("A_log_transposed", "A[n] = -exp(j->A_log[d * N + n]);", "A[n] = -exp(j->A_log[n * j->dim + d]);"),
    ("gate_reads_first_z", "y[t] = zz ? yt * oracle_silu(zz[t]) : yt;",
     "y[t] = zz ? yt * oracle_silu(zz[0]) : yt;"),
    ("initial_state_ignored", "h[n] = j->h0 ? j->h0[chain * N + n] : 0.0;", "h[n] = 0.0;"),
    ("decode_without_dt", "*h = abar * *h + step * B[b * N + n] * x[e];", "*h = abar * *h + B[b * N + n] * x[e];"),
    ("decode_no_gate", "out[e] = z ? yt * oracle_silu(z[e]) : yt;", "out[e] = yt;"),
    ("decode_state_not_decayed", "*h = abar * *h + step * B[b * N + n] * x[e];",
     "*h = *h + step * B[b * N + n] * x[e];"),
    ("decode_C_is_B", "acc += C[b * N + n] * *h;", "acc += B[b * N + n] * *h;"),
    ("decode_skip_dropped", "const double yt = acc + (D ? D[d] : 0.0) * x[e];",
     "const double yt = acc;"),
    ("decode_bias_ignored", "const double raw = dt[e] + (dt_bias ? dt_bias[d] : 0.0);",
     "const double raw = dt[e];"),
    ("softplus_negative_branch_wrong", "return log1p(exp(x));", "return exp(x);"),
    ("dt_reads_first_step", "const double raw = dl[t] + bias;", "const double raw = dl[0] + bias;"),
    ("D_ignores_channel", "const double Dd = j->D ? j->D[d] : 0.0;",
     "const double Dd = j->D ? j->D[0] : 0.0;"),
    ("bias_ignores_channel", "const double bias = j->delta_bias ? j->delta_bias[d] : 0.0;",
     "const double bias = j->delta_bias ? j->delta_bias[0] : 0.0;"),
    ("threads_skip_their_last_chain", "jobs[i].chain_end = chains * (i + 1) / nthreads;",
     "jobs[i].chain_end = chains * (i + 1) / nthreads - (chains > nthreads);"),
    ("reset_ignored", "if (rs && rs[t])", "if (0)"),
    ("reset_after_the_flagged_step", "if (rs && rs[t])", "if (rs && t > 0 && rs[t - 1])"),
    ("reset_one_step_early", "if (rs && rs[t])", "if (rs && t + 1 < L && rs[t + 1])"),
    ("reset_ignores_batch", "j->reset ? j->reset + b * L : NULL", "j->reset ? j->reset : NULL"),
    ("reset_keeps_first_state", "for (int64_t n = 0; n < N; ++n) h[n] = 0.0;",
     "for (int64_t n = 1; n < N; ++n) h[n] = 0.0;"),
    ("bwd_gate_derivative_without_z_term", "s * (1.0 + zz[t] * (1.0 - s))", "s"),
    ("bwd_adjoint_carry_without_decay", "g[n] = a * gn;", "g[n] = gn;"),
    ("bwd_dB_without_dt", "dB[(b * L + t) * N + n] += gn * dt * uc[t];",
     "dB[(b * L + t) * N + n] += gn * uc[t];"),
    ("bwd_dA_uses_updated_state", "dA[d * N + n] += gn * dt * a * hp;",
     "dA[d * N + n] += gn * dt * a * hs[t * N + n];"),
    ("bwd_dA_log_sign", "dA[d * N + n] * -exp(A_log[d * N + n])", "dA[d * N + n] * exp(A_log[d * N + n])"),
    ("bwd_softplus_derivative_missing", "softplus_flag ? ddt / (1.0 + exp(-xr)) : ddt", "ddt"),
    ("bwd_dC_uses_adjoint", "dC[(b * L + t) * N + n] += dy * hs[t * N + n];",
     "dC[(b * L + t) * N + n] += gn * hs[t * N + n];"),
    ("bwd_ddt_without_input_term", "ddt += gn * (A[n] * a * hp + uc[t] * Bb[t * N + n]);",
     "ddt += gn * (A[n] * a * hp);"),
    ("bwd_du_without_skip", "double dut = dy * Dd, ddt = 0.0;", "double dut = 0.0, ddt = 0.0;"),
    ("bwd_du_input_term_without_dt", "dut += gn * dt * Bb[t * N + n];", "dut += gn * Bb[t * N + n];"),
    ("bwd_dD_ignores_gate", "if (dD) dD[d] += dy * uc[t];", "if (dD) dD[d] += go[t] * uc[t];"),
    ("bwd_gate_factor_is_sigmoid", "dy = go[t] * zz[t] * s;", "dy = go[t] * s;"),
    ("bwd_adjoint_drops_later_steps", "const double gn = dy * Cb[t * N + n] + g[n];",
     "const double gn = dy * Cb[t * N + n];"),
    ("bwd_bias_gradient_before_softplus", "if (ddelta_bias) ddelta_bias[d] += dr;",
     "if (ddelta_bias) ddelta_bias[d] += ddt;"),
    ("bwd_reset_ignored", "const double a = (rsb && rsb[t]) ? 0.0 : exp(dt * A[n]);",
     "const double a = exp(dt * A[n]);"),
    ("bwd_reset_one_step_late", "const double a = (rsb && rsb[t]) ? 0.0 : exp(dt * A[n]);",
     "const double a = (rsb && t > 0 && rsb[t - 1]) ? 0.0 : exp(dt * A[n]);"),
    ("bwd_adjoint_ignores_h0",
     "const double gn = dy * Cb[t * N + n] + g[n];\n"
     "                    const double hp = t > 0 ? hs[(t - 1) * N + n] : (hin ? hin[n] : 0.0);",
     "const double gn = dy * Cb[t * N + n] + g[n];\n"
     "                    const double hp = t > 0 ? hs[(t - 1) * N + n] : 0.0;"),
    ("bwd_final_state_gradient_ignored",
     "for (int64_t n = 0; n < N; ++n) g[n] = dlast ? dlast[chain * N + n] : 0.0;",
     "for (int64_t n = 0; n < N; ++n) g[n] = 0.0;"),
    ("bwd_final_state_gradient_from_first_chain",
     "for (int64_t n = 0; n < N; ++n) g[n] = dlast ? dlast[chain * N + n] : 0.0;",
     "for (int64_t n = 0; n < N; ++n) g[n] = dlast ? dlast[n] : 0.0;"),
    ("bwd_dh0_dropped", "dh0[chain * N + n] = g[n];", "dh0[chain * N + n] = 0.0;"),
    ("conv_window_one_step_late", "pre += w[k] * conv_input(xr, st, width, t - (width - 1) + k);",
     "pre += w[k] * conv_input(xr, st, width, t - width + k);"),
    ("conv_taps_reversed", "pre += w[k] * conv_input(xr, st, width, t - (width - 1) + k);",
     "pre += w[width - 1 - k] * conv_input(xr, st, width, t - (width - 1) + k);"),
    ("conv_bias_dropped", "double pre = bias ? bias[d] : 0.0;", "double pre = 0.0;"),
    ("conv_sigmoid_instead_of_silu", "out[row * seqlen + t] = silu_flag ? oracle_silu(pre) : pre;",
     "out[row * seqlen + t] = silu_flag ? 1.0 / (1.0 + exp(-pre)) : pre;"),
    ("conv_state_newest_first", "return st ? st[width - 1 + s] : 0.0;", "return st ? st[-1 - s] : 0.0;"),
    ("conv_state_ignored", "return st ? st[width - 1 + s] : 0.0;", "return 0.0;"),
    ("conv_final_state_shifted", "conv_input(xr, st, width, seqlen - (width - 1) + j);",
     "conv_input(xr, st, width, seqlen - width + j);"),
    ("conv_filter_ignores_channel", "const double *w = weight + d * width;", "const double *w = weight;"),
    ("complex_A_conjugated", "A[n] = -exp(A_log_re[d * N + n]) + I * A_im[d * N + n];",
     "A[n] = -exp(A_log_re[d * N + n]) - I * A_im[d * N + n];"),
    ("complex_A_im_ignored", "A[n] = -exp(A_log_re[d * N + n]) + I * A_im[d * N + n];",
     "A[n] = -exp(A_log_re[d * N + n]);"),
    ("complex_output_imag_part", "const double yt = creal(acc) + (D ? D[d] : 0.0) * ut;",
     "const double yt = cimag(acc) + (D ? D[d] : 0.0) * ut;"),
    ("complex_B_conjugated", "const double complex Bn = B[k] + I * B[k + 1];",
     "const double complex Bn = B[k] - I * B[k + 1];"),
    ("complex_C_pair_swapped", "const double complex Cn = C[k] + I * C[k + 1];",
     "const double complex Cn = C[k + 1] + I * C[k];"),
    ("complex_Bbar_without_dt", "h[n] = cexp(dt * A[n]) * h[n] + dt * Bn * ut;",
     "h[n] = cexp(dt * A[n]) * h[n] + Bn * ut;"),
    ("complex_state_written_conjugated", "last_state[(chain * N + n) * 2 + 1] = cimag(h[n]);",
     "last_state[(chain * N + n) * 2 + 1] = -cimag(h[n]);"),
    ("complex_real_part_of_A_is_minus_A_log",
     "A[n] = -exp(A_log_re[d * N + n]) + I * A_im[d * N + n];",
     "A[n] = -A_log_re[d * N + n] + I * A_im[d * N + n];"),
    ("complex_output_reads_state_before_update",
     "h[n] = cexp(dt * A[n]) * h[n] + dt * Bn * ut;\n                    acc += Cn * h[n];",
     "acc += Cn * h[n];\n                    h[n] = cexp(dt * A[n]) * h[n] + dt * Bn * ut;"),
    ("complex_gate_dropped", "y[chain * L + t] = z ? yt * oracle_silu(z[chain * L + t]) : yt;",
     "y[chain * L + t] = yt;"),
    ("complex_bias_ignored",
     "const double raw = delta[chain * L + t] + (delta_bias ? delta_bias[d] : 0.0);",
     "const double raw = delta[chain * L + t];"),
    ("conv_state_ignores_batch",
     "const double *st = init_state ? init_state + row * (width - 1) : NULL;",
     "const double *st = init_state ? init_state + d * (width - 1) : NULL;"),
    ("conv_activation_always_on", "out[row * seqlen + t] = silu_flag ? oracle_silu(pre) : pre;",
     "out[row * seqlen + t] = oracle_silu(pre);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load(oracle.build(str(src), str(tmp_path / "libmutant.so")))
    failed = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
