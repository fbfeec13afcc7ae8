"""The oracle's pins must be able to fail.

Each case plants one plausible mistake in a temporary copy of the C oracle
source (on the CPU, never in the product), loads the mutant in place of the
real oracle, and checks that at least one pin of tests/test_oracle_pins.py
rejects it.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

MUTANTS = {
    "y_from_previous_state": ("row[n] = alpha * row[n] + u * Bt[n];\n                acc += Ct[n] * row[n];",
                              "acc += Ct[n] * row[n];\n                row[n] = alpha * row[n] + u * Bt[n];"),
    "dropped_D": ("yt[p] = acc + Dh * xt[p];", "yt[p] = acc;"),
    "wrong_sign_of_A": ("const double alpha = exp(dt * Ah);", "const double alpha = exp(-dt * Ah);"),
    "dt_missing_on_input": ("const double u = dt * xt[p];", "const double u = xt[p];"),
    "wrong_group_index": ("const int64_t g = h / (H / G);", "const int64_t g = h % G;"),
    "diag_decay_index": ("st[n] = exp(dt * Ad[n]) * st[n]", "st[n] = exp(dt * Ad[0]) * st[n]"),
    "softplus_before_bias": ("double dt = j->dt[(b * L + t) * Dm + d] + bias;\n        if (j->delta_softplus) dt = softplus(dt);",
                             "double dt = j->dt[(b * L + t) * Dm + d];\n        if (j->delta_softplus) dt = softplus(dt);\n        dt += bias;"),
    "softplus_wrong_branch": ("v + log1p(exp(-v))", "v + log1p(exp(v))"),
    "gate_before_D": ("out *= zt / (1.0 + exp(-zt));", "out = acc * (zt / (1.0 + exp(-zt))) + Dd * xt;"),
    "gate_sigmoid_only": ("out *= zt / (1.0 + exp(-zt));", "out *= 1.0 / (1.0 + exp(-zt));"),
    "conv_window_newest_first": ("for (int64_t k = 0; k + 1 < W; ++k) win[k] = win[k + 1];\n            win[W - 1] = x[b * C + c];",
                                 "for (int64_t k = W - 1; k > 0; --k) win[k] = win[k - 1];\n            win[0] = x[b * C + c];"),
    "conv_bias_dropped": ("double acc = bias ? bias[c] : 0.0;", "double acc = 0.0;"),
    "conv_no_activation": ("out[b * C + c] = act ? silu(acc) : acc;", "out[b * C + c] = acc;"),
    "norm_sum_not_mean": ("const double r = 1.0 / sqrt(ss / (double)group + eps);", "const double r = 1.0 / sqrt(ss + eps);"),
    "norm_gate_after": ("const double g = y[b * D + i] * (z ? silu(z[b * D + i]) : 1.0);\n                ss += g * g;",
                        "const double g = y[b * D + i];\n                ss += g * g;"),
    "bwd_adjoint_not_decayed": ("for (int64_t k = 0; k < PN; ++k) gbar[k] *= alpha;", ""),
    "bwd_dx_without_D": ("dxt[p] = Dh * dyt[p] + dt * gb;", "dxt[p] = dt * gb;"),
    "bwd_ddt_without_decay_term": ("j->ddt[(b * L + t) * H + h] = dalpha * alpha * Ah + xgb;",
                                   "j->ddt[(b * L + t) * H + h] = xgb;"),
    "bwd_dC_from_previous_state": ("c_ += dyt[p] * ht[p * N + n];", "c_ += dyt[p] * hprev[p * N + n];"),
    "bwd_dalpha_from_current_state": ("dalpha += gbar[p * N + n] * hprev[p * N + n];",
                                      "dalpha += gbar[p * N + n] * ht[p * N + n];"),
    "norm_sigmoid_gate": ("static double silu(double v) { return v / (1.0 + exp(-v)); }",
                          "static double silu(double v) { return 1.0 / (1.0 + exp(-v)); }"),
}

PINS = [
    pins.test_A_zero_closed_form, pins.test_single_token_closed_form, pins.test_memoryless_under_strong_decay,
    pins.test_dt_zero_keeps_state, pins.test_lfilter_constant_dt, pins.test_brute_force_tiny,
    pins.test_hand_worked_example, pins.test_quadratic_form_matches_recurrence,
    pins.test_mamba2_equals_mamba1_with_tied_decay, pins.test_diag_lfilter_constant_dt,
    pins.test_diag_delta_bias_and_softplus_reduce_to_transformed_dt, pins.test_diag_softplus_of_large_steps,
    pins.test_diag_z_gate_is_silu_of_z, pins.test_diag_options_single_token_closed_form,
    pins.test_conv_step_sequence_is_numpy_convolve, pins.test_conv_step_continues_from_its_window,
    pins.test_gated_rmsnorm_invariants, pins.test_gated_rmsnorm_gate_ratio_and_eps,
    pins.test_decode_layer_matches_conv_then_prefill_then_norm,
    lambda: pins.test_backward_matches_central_differences(9, None),
    lambda: pins.test_backward_matches_central_differences(70, 40),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found in the oracle source"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new, 1))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(mut), "-o", str(so), "-lm"],
                   check=True)
    oracle._load()  # make sure the real library's argtypes are set up first
    lib = ctypes.CDLL(str(so))
    for fname in ("oracle_ssd_seq", "oracle_ssd_decode", "oracle_diag_seq", "oracle_diag_seq_ex",
                  "oracle_conv1d_step", "oracle_gated_rmsnorm", "oracle_ssd_seq_bwd"):
        getattr(lib, fname).argtypes = getattr(oracle._lib, fname).argtypes
        getattr(lib, fname).restype = ctypes.c_int
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            failed.append(getattr(pin, "__name__", "pin"))
    assert failed, f"no pin rejects the mutant {name}"
