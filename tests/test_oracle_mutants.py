"""The pins have teeth: each plausible mistake planted in a copy of the oracle
(on the CPU, in a temporary build) is caught by at least one pin."""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("dropped_first_term", "for (int k = 0; k < K; ++k) {", "for (int k = 1; k < K; ++k) {"),
    ("wrong_sign", "acc[j] += a * brow[j];", "acc[j] -= a * brow[j];"),
    ("transposed_b", "acc[j] += a * brow[j];", "acc[j] += a * job->Bd[(int64_t)j * K + k];"),
    ("reversed_k_in_a", "job->A[i * (int64_t)K + k]", "job->A[i * (int64_t)K + (K - 1 - k)]"),
    ("subnormal_scale", "mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -23);"),
    ("exponent_bias", "efield - 25", "efield - 24"),
    ("ties_away", "return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;", "return fl + 1.0;"),
    ("overflow_threshold", "if (a >= 65520.0)", "if (a >= 65504.0)"),
    ("subnormal_round", "round_half_even(ldexp(a, 24))", "round_half_even(ldexp(a, 23))"),
    ("lost_carry", "e += 1;", "e += 0;"),
    ("f32_via_f16", "return (float)x;", "return (float)oracle_f16_decode(oracle_f16_round(x));"),
    ("first_row_only", "int64_t i = job->rows[r];", "int64_t i = job->rows[0];"),
    ("start_value_ignored", "for (int j = 0; j < N; ++j) acc[j] = oracle_f16_decode(cin[j]);",
     "for (int j = 0; j < N; ++j) acc[j] = 0.0;"),
    ("add_subtracts", "Z[i] = X[i] + Y[i];", "Z[i] = X[i] - Y[i];"),
    ("add_drops_y", "Z[i] = X[i] + Y[i];", "Z[i] = X[i];"),
    ("start_value_wrong_row", "const uint16_t *cin = (const uint16_t *)job->Cin + i * (int64_t)N;",
     "const uint16_t *cin = (const uint16_t *)job->Cin + r * (int64_t)N;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} must be unique"
    mutated = tmp_path / f"oracle_{name}.c"
    mutated.write_text(src.replace(old, new))
    lib_path = oracle.build(src=str(mutated), out=str(tmp_path / f"lib_{name}.so"))
    lib = oracle.load(lib_path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin caught the planted mistake {name}"
