"""Planted mistakes in copies of the oracle source must each fail some pin.

Every mutant below is a plausible slip in a plain GEMM (a wrong sign, a dropped
term, a transposed operand, a wrong stride, binary32 accumulation, a wrong
rounding rule, a wrong exponent bias).  The test compiles each mutant on the
CPU and runs all pins of tests/test_oracle.py against it; at least one must
fail, which shows the pins would catch that slip in the real oracle.
"""
import os

import pytest

import oracle
import test_oracle

MUTANTS = {
    "sign": ("acc += a * b;", "acc -= a * b;"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    "dropped_first_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    "b_transposed_in_abt": ("? dec[B[j * ldb + k]]", "? dec[B[k * ldb + j]]"),
    "b_transposed_in_ab": (": dec[B[k * ldb + j]]", ": dec[B[j * ldb + k]]"),
    "a_wrong_stride": ("dec[A[i * lda + k]]", "dec[A[i * K + k]]"),
    "accumulate_binary32": ("double acc = 0.0;", "float acc = 0.0f;"),
    "round_toward_zero": ("double q = nearbyint(ldexp(a, fbits - e));", "double q = trunc(ldexp(a, fbits - e));"),
    "ties_away": ("double q = nearbyint(ldexp(a, fbits - e));", "double q = round(ldexp(a, fbits - e));"),
    "f16_bias": ("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
    "subnormal_scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "no_overflow_to_inf": ("if (field >= emax_field) return sign | inf;", "if (field > emax_field) return sign | inf;"),
    "b_k_reversed": ("? dec[B[j * ldb + k]]", "? dec[B[j * ldb + (K - 1 - k)]]"),
    "dtype_table_swapped": ("g_decode[dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_F16]",
                            "g_decode[dtype == ORACLE_BF16 ? ORACLE_F16 : ORACLE_BF16]"),
    "bf16_read_as_f16": ("return dtype == ORACLE_BF16 ? bf16_bits_to_double(bits) : f16_bits_to_double(bits);",
                         "return f16_bits_to_double(bits);"),
    "fp8_e4m3_bias": ("ldexp((double)(8 + f), e - 10)", "ldexp((double)(8 + f), e - 9)"),
    "fp8_e4m3_ieee_nan_rule": ("if (e == 15 && f == 7) return NAN;", "if (e == 15) return NAN;"),
    "fp8_e5m2_subnormal": ("ldexp((double)f, -16)", "ldexp((double)f, -15)"),
    "fp8_alpha_dropped": ("const double d = alpha * acc;", "const double d = acc;"),
    "fp8_b_k_reversed": ("acc += dec[A[i * lda + k]] * dec[B[j * ldb + k]];",
                         "acc += dec[A[i * lda + k]] * dec[B[j * ldb + (K - 1 - k)]];"),
    "fp8_sign": ("acc += dec[A[i * lda + k]] * dec[B[j * ldb + k]];",
                 "acc -= dec[A[i * lda + k]] * dec[B[j * ldb + k]];"),
    "fp8_formats_swapped": ("dec[c] = oracle_fp8_to_double((uint8_t)c, in_fmt);",
                            "dec[c] = oracle_fp8_to_double((uint8_t)c, 1 - in_fmt);"),
    "mx_group_64": ("scale[SA[i * ldsa + k / 32]]", "scale[SA[i * ldsa + k / 64]]"),
    "mx_b_group_16_clamped": ("scale[SB[j * ldsb + k / 32]]",
                              "scale[SB[j * ldsb + (k / 16 < ldsb ? k / 16 : ldsb - 1)]]"),
    "mx_ue8m0_bias": ("return ldexp(1.0, (int)x - 127);", "return ldexp(1.0, (int)x - 128);"),
    "mx_b_scale_dropped": ("dec[B[j * ldb + k]] * scale[SB[j * ldsb + k / 32]]", "dec[B[j * ldb + k]]"),
    "mx_a_scale_first_group_only": ("scale[SA[i * ldsa + k / 32]]", "scale[SA[i * ldsa]]"),
    "mx_a_scale_unpadded_stride": ("scale[SA[i * ldsa + k / 32]]", "scale[SA[i * (K / 32) + k / 32]]"),
    "mx_scale_linear": ("scale[c] = oracle_ue8m0_to_double((uint8_t)c);", "scale[c] = (double)c;"),
    "mx_nan_ignored": ("if (x == 255) return NAN;", "if (x == 255) return 0.0;"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


def _failing_pins(orc):
    failed = []
    for name, fn in test_oracle.PINS.items():
        try:
            fn(orc)
        except AssertionError:
            failed.append(name)
    return failed


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant, mutant_dir):
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
    c_path = os.path.join(mutant_dir, f"{mutant}.c")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.compile_source(c_path, os.path.join(mutant_dir, f"lib{mutant}.so"))
    failed = _failing_pins(oracle.Oracle(so))
    assert failed, f"no pin caught the planted mistake {mutant!r}"
