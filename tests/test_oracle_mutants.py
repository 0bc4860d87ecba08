"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that the
pins in test_oracle_pins.py reject every one of them.  The real oracle source is
never modified: each mutant is compiled from a patched copy in a temporary folder."""
import ctypes
import importlib.util
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "selscan_oracle.c")

# (name, original text, replacement): each original must occur in the source.
MUTANTS = [
    ("drop_D_skip", "const double skip = Dd * ut;", "const double skip = 0.0 * ut;"),
    ("A_sign_flipped", "A[n] = -exp((double)A_log[d * N + n]);", "A[n] = exp((double)A_log[d * N + n]);"),
    ("A_log_transposed", "A[n] = -exp((double)A_log[d * N + n]);",
     "A[n] = -exp((double)A_log[(n % Dm) * N + (d % N)]);"),
    ("b_without_delta", "h[n] = exp(delta * A[n]) * h[n] + delta * (double)B[ib + n] * ut;",
     "h[n] = exp(delta * A[n]) * h[n] + (double)B[ib + n] * ut;"),
    ("decay_without_delta", "h[n] = exp(delta * A[n]) * h[n] + delta * (double)B[ib + n] * ut;",
     "h[n] = exp(A[n]) * h[n] + delta * (double)B[ib + n] * ut;"),
    ("state_not_carried", "h[n] = exp(delta * A[n]) * h[n] + delta * (double)B[ib + n] * ut;",
     "h[n] = exp(delta * A[n]) * 0.0 + delta * (double)B[ib + n] * ut;"),
    ("bias_after_softplus", "oracle_softplus((double)delta_raw[io] + bias)",
     "(oracle_softplus((double)delta_raw[io]) + bias)"),
    ("skip_after_gate", "y_rows[r * L + t] = (acc + skip) * gate;", "y_rows[r * L + t] = acc * gate + skip;"),
    ("gate_is_sigmoid", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("softplus_without_log", "return fmax(x, 0.0) + log1p(exp(-fabs(x)));",
     "return fmax(x, 0.0) + exp(-fabs(x));"),
    ("B_from_previous_step", "const int64_t ib = (b * L + t) * N;",
     "const int64_t ib = (b * L + (t > 0 ? t - 1 : t)) * N;"),
    ("C_replaced_by_B", "const double ch = (double)C[ib + n] * h[n];",
     "const double ch = (double)B[ib + n] * h[n];"),
    ("u_wrong_channel", "const double ut = (double)u[io];",
     "const double ut = (double)u[(b * L + t) * Dm + (Dm - 1 - d)];"),
    ("step_without_decay", "*h = exp(delta * An) * (*h) + delta * xt * (double)B[b * N + n];",
     "*h = (*h) + delta * xt * (double)B[b * N + n];"),
    ("h0_ignored", "for (int64_t n = 0; n < N; ++n) h[n] = h0[row * N + n];",
     "for (int64_t n = 0; n < N; ++n) h[n] = 0.0 * h0[row * N + n];"),
    ("h0_wrong_row", "for (int64_t n = 0; n < N; ++n) h[n] = h0[row * N + n];",
     "for (int64_t n = 0; n < N; ++n) h[n] = h0[((row + 1) % (batch * Dm)) * N + n];"),
    ("h0_scaled", "for (int64_t n = 0; n < N; ++n) h[n] = h0[row * N + n];",
     "for (int64_t n = 0; n < N; ++n) h[n] = 0.5 * h0[row * N + n];"),
    ("h0_not_in_chunked_carry", "double carry = h0 ? h0[row * N + n] : 0.0;", "double carry = 0.0;"),
    ("conv_kernel_flipped", "for (int64_t k = 0; k < K; ++k) acc += (double)w[d * K + k] * e[t + k];",
     "for (int64_t k = 0; k < K; ++k) acc += (double)w[d * K + (K - 1 - k)] * e[t + k];"),
    ("conv_window_off_by_one", "for (int64_t k = 0; k < K; ++k) acc += (double)w[d * K + k] * e[t + k];",
     "for (int64_t k = 0; k < K; ++k) acc += (double)w[d * K + k] * (t + k + 1 < L + K - 1 ? e[t + k + 1] : 0.0);"),
    ("conv_window_ignored", "for (int64_t k = 0; k < K - 1; ++k) e[k] = win_in ? win_in[row * (K - 1) + k] : 0.0;",
     "for (int64_t k = 0; k < K - 1; ++k) e[k] = 0.0 * (win_in ? win_in[row * (K - 1) + k] : 0.0);"),
    ("conv_bias_dropped", "const double bd = bias ? (double)bias[d] : 0.0;",
     "const double bd = bias ? 0.0 * (double)bias[d] : 0.0;"),
    ("conv_act_before_bias", "out[(b * L + t) * Dm + d] = act ? oracle_silu(acc) : acc;",
     "out[(b * L + t) * Dm + d] = act ? oracle_silu(acc - bd) + bd : acc;"),
    ("conv_window_out_stale", "for (int64_t k = 0; k < K - 1; ++k) win_out[row * (K - 1) + k] = e[L + k];",
     "for (int64_t k = 0; k < K - 1; ++k) win_out[row * (K - 1) + k] = e[k];"),
    ("bwd_adjoint_without_decay", "lam[n] = a * l;", "lam[n] = l;"),
    ("bwd_dDelta_decay_sign", "ddel += l * (A[n] * a * hp + (double)B[ib + n] * ut);",
     "ddel += l * (-A[n] * a * hp + (double)B[ib + n] * ut);"),
    ("bwd_softplus_derivative_dropped", "ddelta_raw[io] = ddel * sig_r;", "ddelta_raw[io] = ddel;"),
    ("bwd_du_without_skip", "double dut = Dd * dyh, ddel = 0.0;", "double dut = 0.0 * dyh, ddel = 0.0;"),
    ("bwd_dz_without_yhat", "dz[io] = z ? (double)dy[io] * yhat * dg : 0.0;", "dz[io] = z ? (double)dy[io] * dg : 0.0;"),
    ("bwd_dA_log_chain_dropped", "dA_log[d * N + n] = sA * (-exp((double)A_log[d * N + n]));",
     "dA_log[d * N + n] = sA;"),
    ("bwd_dC_previous_state", "dC[ib + n] += dyh * hs[(t + 1) * N + n];", "dC[ib + n] += dyh * hs[t * N + n];"),
    ("dtproj_W_transposed", "draw += (double)W_dt[d * R + k] * (double)dt_low[(b * L + t) * R + k];",
     "draw += (double)W_dt[k * Dm + d] * (double)dt_low[(b * L + t) * R + k];"),
    ("dtproj_rank_term_dropped", "for (int64_t k = 0; k < R; ++k) draw +=", "for (int64_t k = 1; k < R; ++k) draw +="),
    ("step_bias_dropped",
     "oracle_softplus((double)delta_raw[row] + (delta_bias ? (double)delta_bias[d] : 0.0))",
     "oracle_softplus((double)delta_raw[row])"),
]


def _load_by_path(name, path, search=None):
    spec = importlib.util.spec_from_file_location(name, path, submodule_search_locations=search)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def harness():
    pins = _load_by_path("_oracle_pins_for_mutants", os.path.join(ROOT, "tests", "test_oracle_pins.py"))
    conv = _load_by_path("_oracle_conv_pins_for_mutants", os.path.join(ROOT, "tests", "test_oracle_conv1d.py"))
    bwd = _load_by_path("_oracle_bwd_pins_for_mutants", os.path.join(ROOT, "tests", "test_oracle_bwd.py"))
    dtp = _load_by_path("_oracle_dtproj_pins_for_mutants", os.path.join(ROOT, "tests", "test_oracle_dtproj.py"))
    mod = _load_by_path("_oracle_mutant_pkg", os.path.join(ROOT, "oracle", "__init__.py"),
                        [os.path.join(ROOT, "oracle")])
    battery = [
        pins.test_A_to_zero_is_cumulative_sum,
        pins.test_constant_inputs_geometric_series,
        pins.test_unrolled_sum_form,
        pins.test_skip_only_when_B_or_C_is_zero,
        pins.test_hand_worked_example,
        pins.test_single_step_by_hand,
        pins.test_decode_iterated_equals_forward,
        pins.test_prefix_then_decode_equals_forward,
        pins.test_channel_permutation_and_batch_independence,
        pins.test_linear_in_u_without_gate,
        lambda m: pins.test_chunked_scan_equals_sequential(m, 3),
        pins.test_softplus_textbook,
        pins.test_silu_textbook,
        pins.test_h0_zero_input_is_pure_decay,
        pins.test_h0_with_A_to_zero_adds_to_the_running_sum,
        lambda m: pins.test_h0_split_composition(m, 17),
        pins.test_h0_chunked_equals_sequential,
        pins.test_h0_decode_iterated_equals_forward,
        conv.test_conv1d_matches_numpy_correlate,
        conv.test_conv1d_impulse_response,
        conv.test_conv1d_constant_input_and_left_edge,
        lambda m: conv.test_conv1d_split_composition(m, 11),
        lambda m: conv.test_conv1d_split_composition(m, 2),
        conv.test_conv1d_window_shift_for_short_calls,
        conv.test_conv1d_silu,
        lambda m: bwd.test_bwd_matches_finite_differences(m, True),
        lambda m: bwd.test_bwd_matches_finite_differences(m, False),
        bwd.test_bwd_A_to_zero_closed_form,
        bwd.test_bwd_matches_the_derivative_of_the_unrolled_sum,
        dtp.test_dtproj_exact_projection_matches_plain_forward,
        lambda m: dtp.test_dtproj_general_projection_to_fp32_rounding(m, 4),
    ]
    return mod, battery


def test_unmutated_copy_passes(harness, tmp_path):
    mod, battery = harness
    lib = tmp_path / "orig.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", SRC, "-o", str(lib), "-lm"], check=True)
    mod._lib = mod._configure(ctypes.CDLL(str(lib)))
    for pin in battery:
        pin(mod)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(harness, tmp_path, name, old, new):
    mod, battery = harness
    text = open(SRC).read()
    assert old in text, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(old, new, 1))
    lib = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(src), "-o", str(lib), "-lm"],
                   check=True)
    mod._lib = mod._configure(ctypes.CDLL(str(lib)))
    failures = 0
    for pin in battery:
        try:
            pin(mod)
        except AssertionError:
            failures += 1
    assert failures > 0, f"no pin rejects the planted mistake {name}"
