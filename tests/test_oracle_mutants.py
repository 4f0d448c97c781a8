"""Planted mistakes in copies of the oracle must each be caught by a pin.

Each mutant is a one-place edit of ``oracle/qm_oracle.c`` (a dropped term, a
wrong sign, index or shift, a transposed output, a skipped k-block), compiled
into a temporary library.  The pins of ``oracle_pins.py`` run against it; at
least one must fail, which shows the pins are strong enough to trust the
oracle they pass.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "qm_oracle.c")

MUTANTS = {
    "high_half_reads_low_nibble": ("return (qs[j - 16] >> 4) & 0x0F;", "return qs[j - 16] & 0x0F;"),
    "low_half_reads_high_nibble": ("if (j < 16) return qs[j] & 0x0F;", "if (j < 16) return (qs[j] >> 4) & 0x0F;"),
    "halves_pair_wrong_byte": ("return (qs[j - 16] >> 4) & 0x0F;", "return (qs[31 - j] >> 4) & 0x0F;"),
    "dequant_drops_bias": ("double x = (double)(block_nibble(block, j) - 8) * d;",
                           "double x = (double)(block_nibble(block, j)) * d;"),
    "dequant_bias_7": ("double x = (double)(block_nibble(block, j) - 8) * d;",
                       "double x = (double)(block_nibble(block, j) - 7) * d;"),
    "matmul_drops_bias": ("return (double)(block_nibble(block, j) - 8) * block_scale(block);",
                          "return (double)(block_nibble(block, j)) * block_scale(block);"),
    "scale_big_endian": ("uint16_t bits = (uint16_t)(block[0] | ((uint16_t)block[1] << 8));",
                         "uint16_t bits = (uint16_t)(block[1] | ((uint16_t)block[0] << 8));"),
    "f16_bias_16": ("magnitude = ldexp(1.0 + (double)fraction / 1024.0, exponent - 15);",
                    "magnitude = ldexp(1.0 + (double)fraction / 1024.0, exponent - 16);"),
    "f16_subnormal_shift": ("magnitude = ldexp((double)fraction, -24);",
                            "magnitude = ldexp((double)fraction, -25);"),
    "f16_sign_dropped": ("return sign ? -magnitude : magnitude;", "return magnitude;"),
    "f16_nan_as_inf": ("magnitude = (fraction == 0) ? INFINITY : NAN;", "magnitude = INFINITY;"),
    "quant_offset_1": ("const uint8_t* qs = block + 2;", "const uint8_t* qs = block + 1;"),
    "block_stride_16": ("#define ORACLE_Q4_0_BLOCK_BYTES 18", "#define ORACLE_Q4_0_BLOCK_BYTES 16"),
    "wrong_block_in_row": ("const uint8_t* block = wq + (n * blocks_per_row + b) * ORACLE_Q4_0_BLOCK_BYTES;",
                           "const uint8_t* block = wq + (n * blocks_per_row + (b + 1) % blocks_per_row) * ORACLE_Q4_0_BLOCK_BYTES;"),
    "skip_last_k_block": ("for (int64_t k = 0; k < K; ++k) {\n        double product",
                          "for (int64_t k = 0; k < K - 32; ++k) {\n        double product"),
    "sum_sign_flipped": ("c += product;", "c -= product;"),
    "abs_sum_not_abs": ("s += fabs(product);", "s += product;"),
    "output_transposed": ("entry(A, wq, K, m, n, &C[m * N + n], S ? &S[m * N + n] : NULL);",
                          "entry(A, wq, K, m, n, &C[n * M + m], S ? &S[n * M + m] : NULL);"),
    "activation_row_ignored": ("double product = (double)A[m * K + k] * weight_at(wq, K, n, k);",
                               "double product = (double)A[k] * weight_at(wq, K, n, k);"),
    "weight_row_ignored": ("double product = (double)A[m * K + k] * weight_at(wq, K, n, k);",
                           "double product = (double)A[m * K + k] * weight_at(wq, K, 0, k);"),
    # Q8_0 dequant and quantize, and the binary16 narrowing
    "q8_dequant_unsigned": ("int qs = (int)(int8_t)block[2 + j];", "int qs = (int)block[2 + j];"),
    "q8_dequant_stride_33": ("const uint8_t* block = blob + b * ORACLE_Q8_0_BLOCK_BYTES;",
                             "const uint8_t* block = blob + b * 33;"),
    "q8_divisor_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "q8_ties_to_even": ("double r = round((double)t);", "double r = nearbyint((double)t);"),
    "q8_divides_by_narrowed_d": ("float t = xb[j] / d;",
                                 "float t = xb[j] / (float)oracle_f16_to_double(bits);"),
    "q8_scale_big_endian": ("block[0] = (uint8_t)(bits & 0xFF);\n        block[1] = (uint8_t)(bits >> 8);",
                            "block[1] = (uint8_t)(bits & 0xFF);\n        block[0] = (uint8_t)(bits >> 8);"),
    "q8_max_without_abs": ("float a = fabsf(xb[j]);", "float a = xb[j];"),
    # the product with quantized activations
    "q8act_skips_quantization": ("oracle_dequant_q8_0(q8, K / ORACLE_Q4_0_BLOCK_ELEMS, row);",
                                 "for (int64_t k = 0; k < K; ++k) row[k] = A[m * K + k];"),
    "q8act_every_row_from_row_0": ("for (int64_t m = 0; m < M; ++m) dequantized_row(A, K, m, q8, rows + m * K);\n#ifdef _OPENMP\n#pragma omp parallel for collapse(2)",
                                   "for (int64_t m = 0; m < M; ++m) dequantized_row(A, K, 0, q8, rows + m * K);\n#ifdef _OPENMP\n#pragma omp parallel for collapse(2)"),
    "q8_quants_offset_128": ("block[2 + j] = (uint8_t)(int8_t)q;", "block[2 + j] = (uint8_t)(q + 128);"),
    "q8_no_zero_scale_guard": ("if (d != 0.0f) {", "if (1) {"),
    "q8_no_clamp": ("if (r > 127.0) r = 127.0;", ""),
    "f16_narrow_truncates": ("double m = nearbyint(a / ldexp(1.0, e - 10));",
                             "double m = floor(a / ldexp(1.0, e - 10));"),
    "f16_narrow_overflow_early": ("if (a >= 65520.0)", "if (a > 65504.0)"),
    "f16_narrow_subnormal_shift": ("double m = nearbyint(a / ldexp(1.0, -24));",
                                   "double m = nearbyint(a / ldexp(1.0, -25));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    texts = {f: open(os.path.join(os.path.dirname(SRC), f)).read()
             for f in ("qm_oracle.c", "qm_oracle.h")}
    sites = sum(t.count(before) for t in texts.values())
    assert sites == 1, f"mutation site for {name} not found exactly once"
    for f, t in texts.items():
        (tmp_path / f).write_text(t.replace(before, after))
    lib = oracle.build(str(tmp_path / "qm_oracle.c"), str(tmp_path / "libmutant.so"))
    o = oracle.load(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
