"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Each mutant is a one-line edit of ``oracle.c`` (a dropped term, a wrong sign,
a swapped index, a wrong exponent bias, a wrong rounding), compiled on the CPU
into a temporary directory.  Every edit keeps all memory accesses in bounds.
The pins of ``test_oracle.py`` run against the mutant; at least one must fail.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

GEMM_PINS = [
    pins.test_gemm_identity_both_sides,
    pins.test_gemm_permutation_rows,
    pins.test_gemm_rank1_closed_form,
    pins.test_gemm_integer_exact_against_int64,
    pins.test_gemm_nonsquare_matches_library_matmul,
]
FORMAT_PINS = [
    pins.test_f16_decode_all_patterns,
    pins.test_bf16_decode_all_patterns,
    pins.test_f16_encode_roundtrip_and_ties,
    pins.test_f16_encode_random_and_edges,
]
BF16_PINS = [
    pins.test_bf16_encode_roundtrip_ties_and_random,
    pins.test_gemm_bf16_matches_library_matmul_and_integers,
]
GEMV_PINS = [
    pins.test_gemv_bf16_matches_library_dot,
    pins.test_gemv_bf16_integer_exact_and_layout,
    pins.test_gemv_q8_group_scale_closed_form,
    pins.test_gemv_q8_one_hot_positions,
]

MUTANTS = {
    "bf16_round_down": ("double q = nearbyint(ldexp(a, 7 - E));", "double q = floor(ldexp(a, 7 - E));", BF16_PINS),
    "bf16_bias": ("return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)((int)q - 128));",
                  "return (uint16_t)(sign | (uint16_t)((E + 126) << 7) | (uint16_t)((int)q - 128));", BF16_PINS),
    "gemm_decodes_bf16_as_f16": ("return dtype ? sdt_oracle_bf16_to_f64(v) : sdt_oracle_f16_to_f64(v);",
                                 "return sdt_oracle_f16_to_f64(v);", BF16_PINS),
    "gemm_drops_last_k": ("for (int64_t k = 0; k < K; ++k) {",
                          "for (int64_t k = 0; k < K - 1; ++k) {", GEMM_PINS),
    "gemm_sign": ("acc[j] += a * brow[j];", "acc[j] -= a * brow[j];", GEMM_PINS),
    "gemm_b_row_index": ("const double *brow = Bd + k * N;",
                         "const double *brow = Bd + (K - 1 - k) * N;", GEMM_PINS),
    "gemm_a_col_index": ("double a = sdt_oracle_decode(A[i * K + k], dtype);",
                         "double a = sdt_oracle_decode(A[i * K + (K - 1 - k)], dtype);", GEMM_PINS),
    "f16_bias": ("v = ldexp((double)(f + 1024), e - 25);",
                 "v = ldexp((double)(f + 1024), e - 24);", FORMAT_PINS),
    "f16_subnormal": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);", FORMAT_PINS),
    "f16_round_down": ("double q = nearbyint(ldexp(a, 10 - E));",
                       "double q = floor(ldexp(a, 10 - E));", FORMAT_PINS),
    "bf16_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;", FORMAT_PINS),
    "gemv_w_transposed": ("acc += xd[k] * sdt_oracle_bf16_to_f64(W[n * K + k]);",
                          "acc += xd[k] * sdt_oracle_bf16_to_f64(W[(k % N) * K + (n * K + k) / N % K]);",
                          GEMV_PINS),
    "q8_scale_wrong_group": ("acc += sdt_oracle_f16_to_f64(s[n * n_groups + g]) * part;",
                             "acc += sdt_oracle_f16_to_f64(s[n * n_groups + (g + 1) % n_groups]) * part;",
                             GEMV_PINS),
    "q8_scale_wrong_row": ("acc += sdt_oracle_f16_to_f64(s[n * n_groups + g]) * part;",
                           "acc += sdt_oracle_f16_to_f64(s[((n + 1) % N) * n_groups + g]) * part;",
                           GEMV_PINS),
    "q8_group_boundary": ("for (int64_t k = g * G; k < (g + 1) * G; ++k)",
                          "for (int64_t k = g * G; k < (g + 1) * G - 1; ++k)", GEMV_PINS),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new, checks = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old}"
    mutant_c = tmp_path / "oracle_mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(mutant_c), "-o", str(so), "-lm"])
    prev = oracle._use_library(str(so))
    caught = []
    try:
        for check in checks:
            try:
                check()
            except (AssertionError, ValueError):
                caught.append(check.__name__)
    finally:
        oracle._lib = prev
    assert caught, f"no pin caught mutant {name}"
