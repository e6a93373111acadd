"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that the pins catch every one.  The oracle source itself is never changed:
each mutant is a textual edit of a temporary copy, built with the same flags.
"""
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement).  Only the first occurrence is edited.
MUTANTS = [
    ("dropped_decay", "h[n] = dA * h[n] + dBu;", "h[n] = h[n] + dBu;"),
    ("decay_sign", "const double dA = exp(x);", "const double dA = exp(-x);"),
    ("C_for_B_in_output", "y += C[r + n] * h[n];", "y += B[r + n] * h[n];"),
    ("dropped_delta_in_input", ": delta) : delta;", ": delta) : 1.0;"),
    ("dropped_skip", "y += skip * ut;", ";"),
    ("gate_without_sigmoid", "if (z) y *= oracle_silu(z[i]);",
     "if (z) y *= z[i];"),
    ("sigmoid_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("softplus_as_exp", "return log1p(exp(x));", "return exp(x);"),
    ("softplus_pos_branch", "if (x > 0.0) return x + log1p(exp(-x));",
     "if (x > 0.0) return log1p(exp(-x));"),
    ("A_transposed", "delta * A[d * d_state + n];", "delta * A[n * d_inner + d];"),
    ("BC_ignore_batch", "const int64_t r = (b * L + t) * d_state;",
     "const int64_t r = t * d_state;"),
    ("dropped_bias", "oracle_softplus(dt_raw[i] + bias)",
     "oracle_softplus(dt_raw[i])"),
    ("strictly_causal_output",
     "h[n] = dA * h[n] + dBu;\n            y += C[r + n] * h[n];",
     "y += C[r + n] * h[n];\n            h[n] = dA * h[n] + dBu;"),
    ("skip_index", "const double skip = D ? D[d] : 0.0;",
     "const double skip = D ? D[0] : 0.0;"),
    ("ignored_h0", "h[n] = h0 ? h0[c * d_state + n] : 0.0;", "h[n] = 0.0;"),
    ("decode_state_offset", "state + c * d_state,", "state + d * d_state,"),
    ("segment_transfer_dropped", "a = dA * a;", "a = dA;"),
    ("segment_merge_no_decay",
     "h[n] = a_seg[k * d_state + n] * h[n] + b_seg[k * d_state + n];",
     "h[n] = h[n] + b_seg[k * d_state + n];"),
    ("zoh_ignored", "const double gain = zoh ?", "const double gain = 0 ?"),
    ("zoh_exp_for_expm1", "delta * (expm1(x) / x)", "delta * (exp(x) / x)"),
    ("zoh_gain_without_delta", "delta * (expm1(x) / x)", "(expm1(x) / x)"),
    ("zoh_zero_limit", "(x != 0.0 ? delta * (expm1(x) / x) : delta)",
     "(x != 0.0 ? delta * (expm1(x) / x) : 0.0)"),
    ("zoh_on_decay_too", "const double dA = exp(x);",
     "const double dA = zoh ? expm1(x) : exp(x);"),
    ("decode_ignores_zoh", "b, d, 0, 1, 1, d_inner, d_state, zoh);",
     "b, d, 0, 1, 1, d_inner, d_state, 0);"),
    ("conv_kernel_flipped", "acc += w[d * d_conv + k] * XAT(t - H + k);",
     "acc += w[d * d_conv + (d_conv - 1 - k)] * XAT(t - H + k);"),
    ("conv_no_bias", "double acc = bias ? bias[d] : 0.0;\n            for",
     "double acc = 0.0;\n            for"),
    ("conv_no_silu", "out[(b * L + t) * d_inner + d] = silu ? oracle_silu(acc) : acc;",
     "out[(b * L + t) * d_inner + d] = acc;"),
    ("conv_state_in_reversed", "state_in[c * H + H + (s)]", "state_in[c * H - 1 - (s)]"),
    ("conv_state_out_reversed", "state_out[c * H + j] = XAT(L - H + j);",
     "state_out[c * H + j] = XAT(L - 1 - j);"),
    ("conv_update_no_shift", "st[k] = st[k + 1];", "st[k] = st[k];"),
    ("conv_update_no_append", "if (H > 0) st[H - 1] = x[c];", ";"),
    ("conv_update_window_reversed", "acc += w[d * d_conv + k] * st[k];",
     "acc += w[d * d_conv + k] * st[H - 1 - k];"),
    ("trap_no_previous_term", "(1.0 - lt) * delta * bx[n]", "0.0 * bx[n]"),
    ("trap_weights_swapped", "(1.0 - lt) * delta * bx[n] + lt * delta * B[r + n] * ut",
     "lt * delta * bx[n] + (1.0 - lt) * delta * B[r + n] * ut"),
    ("trap_previous_not_advanced", "bx[n] = B[r + n] * ut;", ";"),
    ("trap_previous_decayed", "(1.0 - lt) * delta * bx[n]", "(1.0 - lt) * delta * dA * bx[n]"),
    ("trap_prev_input_ignored",
     "bx[n] = (u_prev && B_prev) ? B_prev[b * d_state + n] * u_prev[c] : 0.0;\n        }",
     "bx[n] = 0.0;\n        }"),
    ("bwd_no_carry", "dh[n] *= a;", ";"),
    ("bwd_ddelta_sign", "ddelta += da * a * A[d * N + n] + dh[n] * B[r + n] * u[i];",
     "ddelta += -da * a * A[d * N + n] + dh[n] * B[r + n] * u[i];"),
    ("bwd_no_sigmoid", "ddt[i] = ddelta * oracle_sigmoid(x);", "ddt[i] = ddelta;"),
    ("bwd_dC_previous_state", "dC[r + n] += dy * hs[(t + 1) * N + n];",
     "dC[r + n] += dy * hs[t * N + n];"),
    ("bwd_dB_no_delta", "dB[r + n] += dh[n] * delta * u[i];", "dB[r + n] += dh[n] * u[i];"),
    ("bwd_dA_no_delta", "dA[d * N + n] += da * a * delta;", "dA[d * N + n] += da * a;"),
    ("bwd_dz_no_silu_slope", "dz[i] = dout[i] * ys[t] * s * (1.0 + z[i] * (1.0 - s));",
     "dz[i] = dout[i] * ys[t] * s;"),
    ("bwd_dy_ungated", "dy = dout[i] * z[i] * s;", "dy = dout[i];"),
    ("bwd_dlast_ignored", "dh[n] = dlast ? dlast[c * N + n] : 0.0;", "dh[n] = 0.0;"),
    ("bwd_du_no_skip", "double dui = dy * skip, ddelta = 0.0;",
     "double dui = 0.0, ddelta = 0.0;"),
    ("segment_rerun_from_zero", "memcpy(hk, h, (size_t)d_state * sizeof(double));",
     "memset(hk, 0, (size_t)d_state * sizeof(double));"),
]


def _fails_some_pin(orc):
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except Exception:          # an assertion, a NaN comparison, a crash
            return check.__name__
    return None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
    mutated = src.replace(old, new, 1)
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(mutated)
    lib = oracle.build(force=True, src=str(path),
                       out=str(tmp_path / f"liboracle_{name}.so"))
    caught_by = _fails_some_pin(oracle.Oracle(lib))
    assert caught_by is not None, f"no pin catches mutant {name}"
