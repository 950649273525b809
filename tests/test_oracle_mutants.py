"""CPU mutation test: planted mistakes in the oracle's C source must fail a pin.

Each mutant is a copy of oracle/gemm_oracle.c with one textual change (a
dropped term, a wrong sign, a transposed index, a reordered epilogue, a
wrong rounding...), compiled into a temporary directory.  The pins of
oracle_pins.py must reject every one of them; a mutant that passes all pins
would mean the pins leave that part of the oracle unchecked.
"""
import os
import tempfile

import pytest

import oracle
from tests import oracle_pins

MUTANTS = [
    ("dropped_term", "s += a * bv;", "if (k != K / 2) s += a * bv;"),
    ("bias_sign", "y += (double)bias[j];", "y -= (double)bias[j];"),
    ("transposed_b", "b_layout == OR_B_KN ? k * ldb + j : j * ldb + k);\n        s += a * bv;",
     "b_layout == OR_B_KN ? j * ldb + k : k * ldb + j);\n        s += a * bv;"),
    ("dropped_beta", "y += beta * (double)R[", "y += (double)R["),
    ("act_before_bias",
     "            if (bias)\n                y += (double)bias[j];\n            y = oracle_act(act, y);",
     "            y = oracle_act(act, y);\n            if (bias)\n                y += (double)bias[j];"),
    ("gelu_scale", "erf(y / sqrt(2.0))", "erf(y / 2.0)"),
    ("round_half_up", "nearbyint(x / quantum)", "floor(x / quantum + 0.5)"),
    ("f16_exponent", "ex - 25", "ex - 24"),
    ("bf16_precision", "round_rne(x, 8, -126", "round_rne(x, 7, -126"),
    ("sabs_signed", "sa += fabs(a * bv);", "sa += a * bv;"),
    ("ignores_lda", "load_elem(Abat, dtype, i * lda + k);\n        double bv",
     "load_elem(Abat, dtype, i * K + k);\n        double bv"),
    ("residual_batch", "R[b * stride_r + i * ldr + j];\n            int64_t o",
     "R[i * ldr + j];\n            int64_t o"),
    ("freivalds_x", "s += bv * x[j];", "s += bv;"),
    ("dropped_alpha", "double y = alpha * s;", "double y = s;"),
    ("relu_abs", "y > 0.0 ? y : 0.0", "y > 0.0 ? y : -y"),
    ("f16_subnormal", "ldexp((double)fr, -24)", "ldexp((double)fr, -25)"),
    ("sample_rows", "int64_t i = rows ? rows[r] : r;", "int64_t i = r;"),
    # row softmax
    ("softmax_no_bias", "t[j] = alpha * s + (bias ? (double)bias[j] : 0.0);", "t[j] = alpha * s;"),
    ("softmax_no_max", "z += exp(t[j] - m);", "z += exp(t[j]);"),
    ("softmax_norm", "double y = exp(t[j] - m) / z;", "double y = exp(t[j] - m) / (z + 1e-3);"),
    ("softmax_sampled_cols", "double* t = (double*)malloc(sizeof(double) * (size_t)(2 * N + 1));",
     "N = ncols; double* t = (double*)malloc(sizeof(double) * (size_t)(2 * N + 1));"),
    ("softmax_alpha_late", "t[j] = alpha * s + (bias", "t[j] = s + (bias"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(source, name, old, new, tmp_path):
    assert source.count(old) == 1, f"mutation site for {name} not unique / not found"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    lib = oracle.compile_oracle(str(src), str(tmp_path / f"lib{name}.so"))
    mutant = oracle.Oracle(lib)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mutant)
        except Exception as e:     # AssertionError, or a rejected argument
            caught.append(check.__name__)
    assert caught, f"mutant {name} passed every pin"
