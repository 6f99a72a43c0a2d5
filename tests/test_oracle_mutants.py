"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle.c (on the CPU), builds it, and
runs the pin suites (test_oracle.py, test_oracle_router.py,
test_oracle_epilogue.py) against it in a
subprocess: they must fail.  The real oracle passing the same suites is those
files themselves.
"""
import os
import subprocess
import sys
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "drop_last_k": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k < K - 1; ++k)"),
    "skip_first_k": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    "sign_error": ("total += oracle_bf16_to_double(X[m * K + k])",
                   "total -= oracle_bf16_to_double(X[m * K + k])"),
    "fp32_accumulator": ("double total = 0.0;", "float total = 0.0f;"),
    "w_layout_ignored": ("w_layout == 0 ? W[n * K + k] : W[k * N + n]", "W[n * K + k]"),
    "w_transposed": ("w_layout == 0 ? W[n * K + k] : W[k * N + n]",
                     "w_layout == 0 ? W[k * N + n] : W[n * K + k]"),
    "x_reversed": ("X[m * K + k])", "X[m * K + (K - 1 - k)])"),
    "bias_twice": ("total += oracle_bf16_to_double(bias[n]);",
                   "total += 2.0 * oracle_bf16_to_double(bias[n]);"),
    "bias_dropped": ("if (bias)\n", "if (0)\n"),
    "decode_shift": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "output_transposed": ("Y[m * N + n] = cell", "Y[n * M + m] = cell"),
    # fp32 router weights: rounding, the high/low split, the fp32-weight product.
    "rne_truncates": ("u += 0x7FFFu + keep_odd;", "u += 0u * keep_odd;"),
    "rne_ties_away": ("u += 0x7FFFu + keep_odd;", "u += 0x8000u + 0u * keep_odd;"),
    "low_from_weight": ("const float r = W[i] - h32;", "const float r = W[i] + 0.0f * h32;"),
    "low_dropped": ("L[i] = oracle_f32_to_bf16(r);", "L[i] = 0;"),
    "f32w_rounded_to_bf16": (
        "const double w = (double)(w_layout == 0 ? W[n * K + kk] : W[kk * N + n]);",
        "const double w = oracle_bf16_to_double(oracle_f32_to_bf16("
        "w_layout == 0 ? W[n * K + kk] : W[kk * N + n]));"),
    "f32w_layout_ignored": ("(w_layout == 0 ? W[n * K + kk] : W[kk * N + n])", "(W[n * K + kk])"),
    # Fused epilogues: GELU's definition and where it applies.
    "gelu_no_half": ("return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));",
                     "return 1.0 * x * (1.0 + erf(x / sqrt(2.0)));"),
    "gelu_scale_two": ("return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));",
                       "return 0.5 * x * (1.0 + erf(x / 2.0));"),
    "gelu_sign": ("return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));",
                  "return 0.5 * x * (1.0 - erf(x / sqrt(2.0)));"),
    "activation_ignored": ("if (act == 1)\n", "if (act == 7)\n"),
    "silu_sign": ("return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    "silu_no_x": ("return x / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(-x));"),
    "swiglu_gates_up": ("out[i] = oracle_silu(gate[i]) * up[i];", "out[i] = gate[i] * oracle_silu(up[i]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_fail_on_mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found in oracle.c"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mutant.c")
        so = os.path.join(d, "mutant.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                        "-o", so, c, "-lm"], check=True)
        env = dict(os.environ, ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                            os.path.join(HERE, "test_oracle.py"),
                            os.path.join(HERE, "test_oracle_router.py"),
                            os.path.join(HERE, "test_oracle_epilogue.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
