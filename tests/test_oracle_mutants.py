"""Planted mistakes in the oracle must fail at least one pin.

Each mutant is a textual edit of a copy of oracle/ssm_oracle.c (a dropped term, a wrong
sign, a wrong or transposed index, the state read before its update, ...), compiled with
gcc into a temporary library; every pin of tests/oracle_pins.py is run against it and at
least one must raise. Runs on the CPU only.
"""
import os
import tempfile

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

# (name, [(old, new), ...]) -- each old string must occur in the source
MUTANTS = [
    ("A_sign", [("double A_bar = exp(dt * A[n]);", "double A_bar = exp(-dt * A[n]);")]),
    ("dropped_step_on_B", [("double B_bar = dt * B[n * L + t];", "double B_bar = B[n * L + t];")]),
    ("B_C_transposed", [("double B_bar = dt * B[n * L + t];", "double B_bar = dt * C[n * L + t];")]),
    ("time_reversed_B", [("double B_bar = dt * B[n * L + t];", "double B_bar = dt * B[n * L + (L - 1 - t)];")]),
    ("read_before_update", [
        ("h[n] = A_bar * h[n] + B_bar * x;\n            hm[n]",
         "double hprev = h[n];\n            h[n] = A_bar * h[n] + B_bar * x;\n            hm[n]"),
        ("acc += h[n] * C[n * L + t];", "acc += hprev * C[n * L + t];")]),
    ("dropped_D", [("double yt = acc + (has_D ? x * Dval : 0.0);", "double yt = acc;")]),
    ("no_softplus", [("if (use_softplus) dt = softplus(dt);", "(void)use_softplus;")]),
    ("bias_after_softplus", [
        ("double dt = delta[t] + (has_bias ? bias : 0.0);\n        if (use_softplus) dt = softplus(dt);",
         "double dt = delta[t];\n        if (use_softplus) dt = softplus(dt);\n        dt += (has_bias ? bias : 0.0);")]),
    ("gate_is_sigmoid", [("static double silu(double v) { return v / (1.0 + exp(-v)); }",
                          "static double silu(double v) { return 1.0 / (1.0 + exp(-v)); }")]),
    ("C_wrong_time", [("acc += h[n] * C[n * L + t];", "acc += h[n] * C[n * L + (t > 0 ? t - 1 : 0)];")]),
    ("decode_A_index", [("double A_bar = exp(dt[bd] * A[d * N + n]);", "double A_bar = exp(dt[bd] * A[n]);")]),
    ("decode_B_batch", [("double B_bar = dt[bd] * B[b * N + n];", "double B_bar = dt[bd] * B[n];")]),
    ("decode_no_D", [("double yt = acc + (Dskip ? x[bd] * Dskip[d] : 0.0);", "double yt = acc;")]),
    ("h0_ignored", [("h[n] = h0 ? h0[n] : 0.0;", "h[n] = 0.0;")]),
    ("zoh_factor_exp_not_expm1", [("return x == 0.0 ? 1.0 : expm1(x) / x;", "return x == 0.0 ? 1.0 : exp(x) / x;")]),
    ("zoh_factor_missing_divide", [("return x == 0.0 ? 1.0 : expm1(x) / x;", "return x == 0.0 ? 1.0 : expm1(x);")]),
    ("zoh_ignored_in_scan", [("if (zoh) B_bar *= zoh_factor(dt * A[n]);", "(void)zoh;")]),
    ("conv_kernel_reversed", [("if (s >= 0) acc += w[c * K + k] * x[c * L + s];",
                               "if (s >= 0) acc += w[c * K + (K - 1 - k)] * x[c * L + s];")]),
    ("conv_padding_off_by_one", [("const int64_t s = t - (K - 1) + k;", "const int64_t s = t - K + k;")]),
    ("conv_bias_dropped", [("double acc = cb ? cb[c] : 0.0;", "double acc = 0.0;")]),
    ("zoh_ignored_in_decode", [("if (zoh) B_bar *= zoh_factor(dt[bd] * A[d * N + n]);", "(void)zoh;")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, edits, tmp_path):
    with open(SRC) as f:
        src = f.read()
    for old, new in edits:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new, 1)
    c = tmp_path / f"mut_{name}.c"
    c.write_text(src)
    so = oracle.compile_oracle(str(c), str(tmp_path / f"libmut_{name}.so"))
    lib = oracle.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_source_passes_every_pin(tmp_path):
    so = oracle.compile_oracle(SRC, str(tmp_path / "libclean.so"))
    lib = oracle.load(so)
    for pin in oracle_pins.ALL_PINS:
        pin(lib)
