"""Plant plausible mistakes in the oracle's C source, on the CPU, and check that the pins catch them.

Each mutant is a one-line textual change of ``oracle/oracle.c`` (a dropped term, a wrong sign or
index, a transposed operand, a misplaced bias), compiled to a temporary library that replaces the
oracle's for the duration of one check.  A mutant passes the check only if at least one pin fails
on it: a pin of ``test_oracle_pins.py`` for the forward scan and the decode step, a pin of
``test_oracle_grad_pins.py`` for the exact zero-order hold and the gradients.
"""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_conv_pins as cpins
import test_oracle_grad_pins as gpins
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "readout_uses_B": ("acc += widen(C, bc, in_dtype) * h[n];", "acc += widen(B, bc, in_dtype) * h[n];"),
    "skip_term_dropped": ("double y = acc + Dd * x;", "double y = acc;"),
    "A_sign_flipped": ("const double Abar = exp(dt * a_n[n]);", "const double Abar = exp(-dt * a_n[n]);"),
    "euler_A": ("const double Abar = exp(dt * a_n[n]);", "const double Abar = 1.0 + dt * a_n[n];"),
    "Bbar_missing_delta": ("const double Bbar_x = bbar_factor(dt, a_n[n], zoh) * widen(B, bc, in_dtype) * x;",
                           "const double Bbar_x = widen(B, bc, in_dtype) * x;"),
    "BC_transposed": ("const long long bc = ((long long)b * dstate + n) * seqlen + t;",
                      "const long long bc = ((long long)b * seqlen + t) * dstate + n;"),
    "BC_batch_ignored": ("const long long bc = ((long long)b * dstate + n) * seqlen + t;",
                         "const long long bc = ((long long)0 * dstate + n) * seqlen + t;"),
    "A_channel_ignored": ("a_n[n] = (double)A[(long long)d * dstate + n];", "a_n[n] = (double)A[n];"),
    "readout_before_update": ("h[n] = Abar * h[n] + Bbar_x;\n                acc += widen(C, bc, in_dtype) * h[n];",
                              "acc += widen(C, bc, in_dtype) * h[n];\n                h[n] = Abar * h[n] + Bbar_x;"),
    "bias_after_softplus": ("double d = raw + bias;\n    return softplus_flag ? softplus(d) : d;",
                            "return softplus_flag ? softplus(raw) + bias : raw + bias;"),
    "gate_is_sigmoid": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "softplus_overflows": ("if (x > 0.0) return x + log1p(exp(-x));", "if (x > 1e300) return x;"),
    "step_skip_dropped": ("double y = acc + (D ? (double)D[d] : 0.0) * x;", "double y = acc;"),
    "step_A_sign": ("const double Abar = exp(dt * a);", "const double Abar = exp(-dt * a);"),
    "bf16_widen_wrong_shift": ("((const uint16_t*)p)[i]) << 16;", "((const uint16_t*)p)[i]) << 15;"),
}

# Mistakes in the exact zero-order hold and in the reverse-mode gradients, caught by the pins of
# tests/test_oracle_grad_pins.py.
GRAD_MUTANTS = {
    "zoh_missing_division": ("return expm1(dt * a) / a;", "return expm1(dt * a);"),
    "zoh_exp_not_expm1": ("return expm1(dt * a) / a;", "return exp(dt * a) / a;"),
    "grad_C_uses_adjoint": ("gC[n * L + t] += e * h_t[n];", "gC[n * L + t] += lam * h_t[n];"),
    "grad_B_missing_x": ("gB[n * L + t] += lam * k * x;", "gB[n * L + t] += lam * k;"),
    "grad_dt_drops_decay_term": ("gdt += lam * (a_n[n] * decay * h_prev[n] + dk_ddt * Bv * x);",
                                 "gdt += lam * (dk_ddt * Bv * x);"),
    "grad_A_uses_new_state": ("gA[n] += lam * (dt * decay * h_prev[n] + dk_da * Bv * x);",
                              "gA[n] += lam * (dt * decay * h_t[n] + dk_da * Bv * x);"),
    "adjoint_not_decayed": ("mu[n] = lam * decay;", "mu[n] = lam;"),
    "gate_grad_is_sigmoid": ("return sg * (1.0 + z * (1.0 - sg));", "return sg;"),
    "softplus_grad_dropped": ("const double gs = softplus_flag ? gdt * softplus_grad(s) : gdt;",
                              "const double gs = gdt;"),
    "skip_grad_dropped": ("double gx = e * Dd, gdt = 0.0;", "double gx = 0.0, gdt = 0.0;"),
    "gate_not_in_adjoint": ("const double e = dy_rows[i * L + t] * gate;",
                            "const double e = dy_rows[i * L + t];"),
    "zoh_dk_da_sign": ("dk_da = (dt * a_n[n] * decay - expm1(dt * a_n[n])) / (a_n[n] * a_n[n]);",
                       "dk_da = (expm1(dt * a_n[n]) - dt * a_n[n] * decay) / (a_n[n] * a_n[n]);"),
    "zoh_dk_ddt_euler": ("dk_ddt = decay;", "dk_ddt = 1.0;"),
    "zoh_zero_A_dk_da": ("dk_da = 0.5 * dt * dt;", "dk_da = dt * dt;"),
}

# Mistakes in the causal convolution, caught by the pins of tests/test_oracle_conv_pins.py.
CONV_MUTANTS = {
    "conv_taps_reversed": ("const long long s = t - (K - 1) + k;", "const long long s = t - k;"),
    "conv_previous_inputs_ignored": ("else if (x_prev_rows)", "else if (0)"),
    "conv_previous_inputs_reversed": ("xv = x_prev_rows[i * (K - 1) + (K - 1) + s];",
                                      "xv = x_prev_rows[i * (K - 1) - 1 - s];"),
    "conv_bias_dropped": ("double acc = conv_bias ? (double)conv_bias[d] : 0.0;", "double acc = 0.0;"),
    "conv_activation_dropped": ("u_rows[i * seqlen + t] = act_silu ? silu(acc) : acc;",
                                "u_rows[i * seqlen + t] = acc;"),
}

CONV_PINS = [
    lambda: cpins.test_conv_matches_numpy_convolve(4),
    cpins.test_conv_activation_is_silu,
    lambda: cpins.test_split_sequence_with_previous_inputs(3),
]

GRAD_PINS = [
    lambda: gpins.test_gradients_match_finite_differences("all_inputs", "simple"),
    lambda: gpins.test_gradients_match_finite_differences("all_inputs", "zoh"),
    lambda: gpins.test_gradients_match_finite_differences("bare", "zoh"),
    gpins.test_zoh_gradients_at_zero_A,
    gpins.test_zoh_matches_numerical_ode,
]

PINS = [
    lambda: pins.test_lti_equals_convolution(1, 16, 4, 64),
    pins.test_lti_tiny_workload_recipe,
    lambda: pins.test_scalar_closed_form_time_varying(1),
    lambda: pins.test_scalar_closed_form_time_varying(4),
    pins.test_closed_form_without_softplus_and_with_initial_state,
    pins.test_single_step_formula,
    pins.test_softplus_and_bias_against_logaddexp,
    pins.test_gate_against_expit,
    pins.test_delta_zero_keeps_state_bit_for_bit,
    pins.test_delta_zero_scan_gives_skip_only,
    pins.test_huge_delta_is_memoryless,
    pins.test_linear_in_u,
    pins.test_decode_steps_equal_scan,
    pins.test_bf16_widening_matches_fp32,
]


def _compile(src_text, out_dir):
    c = os.path.join(out_dir, "mut.c")
    so = os.path.join(out_dir, "libmut.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           "-ffp-contract=off", "-o", so, c, "-lm"])
    return so


def _caught(old, new, pins_to_run, monkeypatch):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutant anchor not found: {old!r}"
    mutated = src.replace(old, new)
    with tempfile.TemporaryDirectory() as td:
        so = _compile(mutated, td)
        mut = ctypes.CDLL(so)
        for fn, argtypes in oracle.SIGNATURES.items():
            getattr(mut, fn).restype = ctypes.c_int
            getattr(mut, fn).argtypes = argtypes
        monkeypatch.setattr(oracle, "_lib", mut)
        caught = []
        for pin in pins_to_run:
            try:
                pin()
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(pin)
                break
        return caught


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    old, new = MUTANTS[name]
    assert _caught(old, new, PINS, monkeypatch), f"no pin caught mutant {name}"


@pytest.mark.parametrize("name", sorted(GRAD_MUTANTS))
def test_grad_pins_catch_mutant(name, monkeypatch):
    old, new = GRAD_MUTANTS[name]
    assert _caught(old, new, GRAD_PINS, monkeypatch), f"no pin caught mutant {name}"


@pytest.mark.parametrize("name", sorted(CONV_MUTANTS))
def test_conv_pins_catch_mutant(name, monkeypatch):
    old, new = CONV_MUTANTS[name]
    assert _caught(old, new, CONV_PINS, monkeypatch), f"no pin caught mutant {name}"
