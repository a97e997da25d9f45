"""Planted mistakes: each broken copy of the oracle must fail at least one pin.

The mistakes are applied to a temporary copy of ``oracle/ssm_oracle.c`` and
compiled on the CPU; the committed oracle is never modified. The list covers
the plausible slips named for the oracle: a dropped term, a wrong sign, a wrong
index, a transposed operand, a wrong softplus or discretisation.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

# name -> (text in the source, replacement); each text must occur in the source.
MUTANTS = {
    "bbar_without_dt": ("return phi * dt * B_n;", "return phi * B_n;"),
    "A_positive": ("A[n] = -exp(A_log[d * dstate + n]);", "A[n] = exp(A_log[d * dstate + n]);"),
    "C_replaced_by_B": ("y += C[j + n] * h[n];", "y += B[j + n] * h[n];"),
    "D_skip_dropped": ("y += D[d] * u[i];                                         /* D skip */",
                       "y += 0.0 * D[d] * u[i];"),
    "gate_without_sigmoid": ("return z / (1.0 + exp(-z));", "return z;"),
    "softplus_wrong_sign": ("return fmax(x, 0.0) + log1p(exp(-fabs(x)));",
                            "return fmax(x, 0.0) + log1p(exp(-x));"),
    "zoh_uses_exp_not_expm1": ("expm1(dA) / dA", "exp(dA) / dA"),
    "readout_before_update": (
        "            h[n] = abar * h[n] + bbar * u[i];                         /* recurrence */\n"
        "            y += C[j + n] * h[n];                                     /* y = C h */",
        "            y += C[j + n] * h[n];\n"
        "            h[n] = abar * h[n] + bbar * u[i];"),
    "B_index_off_by_one_step": ("oracle_bbar(dt, A[n], B[j + n], variant)",
                                "oracle_bbar(dt, A[n], B[(t > 0 ? j - dstate : j) + n], variant)"),
    "bias_ignored": ("const double bias = delta_bias ? delta_bias[d] : 0.0;",
                     "const double bias = 0.0;"),
    "decode_A_index": ("const double A_n = -exp(A_log[d * dstate + n]);",
                       "const double A_n = -exp(A_log[n]);"),
    "decode_state_not_decayed": ("*h = abar * (*h) + bbar * u[i];", "*h = (*h) + bbar * u[i];"),
    # the decode step ignores its variant flag (always zero-order hold)
    "decode_variant_ignored": ("const double bbar = oracle_bbar(dt, A_n, B[b * dstate + n], variant);",
                               "const double bbar = oracle_bbar(dt, A_n, B[b * dstate + n], 0);"),
    # the A -> 0 limit of the input matrix taken as 0 instead of dt B
    "zoh_limit_dropped": ("double phi = (dA == 0.0) ? 1.0 : expm1(dA) / dA;",
                          "double phi = (dA == 0.0) ? 0.0 : expm1(dA) / dA;"),
    "conv_taps_reversed": ("acc += w[d * width + k] * x[(b * seqlen + ts) * dim + d];",
                           "acc += w[d * width + (width - 1 - k)] * x[(b * seqlen + ts) * dim + d];"),
    "conv_without_silu": ("u[(b * seqlen + t) * dim + d] = oracle_silu(acc);",
                          "u[(b * seqlen + t) * dim + d] = acc;"),
    # circular instead of causal zero padding (every index stays inside x)
    "conv_circular_padding": ("const long ts = t - (width - 1) + k;",
                              "const long ts = (t - (width - 1) + k + seqlen) % seqlen;"),
    # backward
    "bwd_dphi_series_coefficient": ("0.5 + s * (1.0 / 3.0 +", "0.5 + s * (1.0 / 4.0 +"),
    "bwd_state_adjoint_not_decayed": ("hbar[n] *= abar; /* to h_prev */", "/* adjoint not carried */"),
    "bwd_abar_adjoint_uses_h_t": ("const double abar_bar = hbar[n] * h_prev;",
                                  "const double abar_bar = hbar[n] * h_t;"),
    "bwd_silu_derivative_is_sigmoid": ("dout[i] * ys[t] * sg * (1.0 + z[i] * (1.0 - sg))", "dout[i] * ys[t] * sg"),
    "bwd_softplus_derivative_sign": ("dtbar * oracle_sigmoid(delta[i] + bias_d)",
                                     "dtbar * oracle_sigmoid(-(delta[i] + bias_d))"),
    "bwd_A_log_chain_sign": ("Abar_acc[n] * A[n]; /* A = -exp(A_log) */", "Abar_acc[n] * -A[n];"),
    "bwd_dt_through_bbar_dropped": ("dtbar += bbar_bar * abar * B_tn;", "dtbar += 0.0;"),
    "bwd_D_path_to_u_dropped": ("ubar += ybar * D[d];", "ubar += 0.0;"),
    "bwd_dC_uses_h_prev": ("dC[j + n] += ybar * h_t;", "dC[j + n] += ybar * h_prev;"),
    "bwd_u_through_state_dropped": ("ubar += hbar[n] * bbar;", "ubar += 0.0 * bbar;"),
    "bwd_readout_adjoint_dropped": ("hbar[n] += ybar * C[j + n];", "hbar[n] += 0.0 * C[j + n];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    text, repl = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(text) == 1, f"mutant {name}: anchor text not found once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(text, repl))
    lib = oracle.OracleLib(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    failed = []
    for pin, (fn, tol) in PINS.items():
        try:
            err = fn(lib)
        except Exception:          # a crash or NaN also counts as caught
            failed.append(pin)
            continue
        if not err <= tol:
            failed.append(pin)
    assert failed, f"planted mistake {name} passed every pin"
