"""The CPU oracle against its pins, and the pins against planted mistakes.

A pin is only worth something if a plausible mistake in the oracle breaks it.
``test_planted_mistake_is_caught`` copies the oracle's C source, plants one
mistake (a dropped term, a wrong sign, a wrong index or stride, a transposed
output, a wrong BF16 decode, FP32 accumulation), builds the copy on the CPU and
requires that at least one pin fails on it. The real oracle is never modified.
"""
import os

import numpy as np
import pytest

from oracle import oracle
from tests import oracle_pins

MUTATIONS = {
    "drop_last_term": ("for (int64_t k = 0; k < K; ++k) {\n                double term",
                       "for (int64_t k = 0; k < K - 1; ++k) {\n                double term"),
    "drop_first_term": ("for (int64_t k = 0; k < K; ++k) {\n                double term",
                        "for (int64_t k = 1; k < K; ++k) {\n                double term"),
    "wrong_sign": ("            acc += term;\n                mag",
                   "            acc -= term;\n                mag"),
    "row_stride_K": ("const uint16_t *wn = W + n * ldw;\n            double acc",
                     "const uint16_t *wn = W + n * K;\n            double acc"),
    "x_stride_ldw": ("const uint16_t *xb = x + b * K;\n        for",
                     "const uint16_t *xb = x + b * ldw;\n        for"),
    "signed_scale": ("mag += term < 0.0 ? -term : term;\n            }\n            y[",
                     "mag += term;\n            }\n            y["),
    "transposed_y": ("y[b * N + n] = acc;", "y[n * B + b] = acc;"),
    "bf16_shift": ("((uint32_t)h) << 16", "((uint32_t)h) << 15"),
    "fp32_accumulate": ("double acc = 0.0;\n            double mag = 0.0;\n            for (int64_t k = 0; k < K; ++k) {\n                double term",
                        "float acc = 0.0f;\n            double mag = 0.0;\n            for (int64_t k = 0; k < K; ++k) {\n                double term"),
    "operand_swap_W_for_x": ("bf16_to_double(wn[k]) * bf16_to_double(xb[k]);\n                acc",
                             "bf16_to_double(wn[k]) * bf16_to_double(wn[k]);\n                acc"),
    "rms_no_eps": ("1.0 / sqrt(sq / (double)K + eps)", "1.0 / sqrt(sq / (double)K)"),
    "rms_sum_not_mean": ("1.0 / sqrt(sq / (double)K + eps)", "1.0 / sqrt(sq + eps)"),
    "rms_no_sqrt": ("1.0 / sqrt(sq / (double)K + eps)", "1.0 / (sq / (double)K + eps)"),
    "rms_abs_not_square": ("            sq += v * v;", "            sq += v < 0.0 ? -v : v;"),
    "rms_scale_unscaled": ("            s[b * N + n] *= rb;\n", ""),
    "rms_mean_over_ldw": ("1.0 / sqrt(sq / (double)K + eps)", "1.0 / sqrt(sq / (double)ldw + eps)"),
    "w4_odd_even_swapped": ("int shift = (i % 2 == 0) ? (int)(4 * (i / 2)) : (int)(16 + 4 * (i / 2));",
                            "int shift = (i % 2 == 1) ? (int)(4 * (i / 2)) : (int)(16 + 4 * (i / 2));"),
    "w4_no_zero_point": ("return (double)(code - 8) *", "return (double)(code) *"),
    "w4_group_64": ("bf16_to_double(S[n * lds + k / group]);", "bf16_to_double(S[n * lds + k / 64]);"),
    "w4_row_stride_half_k": ("const uint8_t *p = Wq + n * ldq + 4 * (k / 8);",
                             "const uint8_t *p = Wq + n * (lds * 64) + 4 * (k / 8);"),
    "w4_scale_row_0": ("bf16_to_double(S[n * lds + k / group]);", "bf16_to_double(S[k / group]);"),
    "w4_big_endian": ("uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);",
                      "uint32_t word = (uint32_t)p[3] | ((uint32_t)p[2] << 8) | ((uint32_t)p[1] << 16) | ((uint32_t)p[0] << 24);"),
    "fp8_bias_8": ("else mag8 = ldexp(1.0 + (double)m8 / 8.0, e8 - 7);",
                   "else mag8 = ldexp(1.0 + (double)m8 / 8.0, e8 - 8);"),
    "fp8_subnormal_exponent": ("if (e8 == 0) mag8 = ldexp((double)m8 / 8.0, -6);",
                               "if (e8 == 0) mag8 = ldexp((double)m8 / 8.0, -7);"),
    "fp8_subnormal_implicit_one": ("if (e8 == 0) mag8 = ldexp((double)m8 / 8.0, -6);",
                                   "if (e8 == 0) mag8 = ldexp(1.0 + (double)m8 / 8.0, -6);"),
    "fp8_sign_dropped": ("return (c & 0x80) ? -mag8 : mag8;", "return mag8;"),
    "fp8_mantissa_over_16": ("else mag8 = ldexp(1.0 + (double)m8 / 8.0, e8 - 7);",
                             "else mag8 = ldexp(1.0 + (double)m8 / 16.0, e8 - 7);"),
    "fp8_no_row_scale": ("e4m3_to_double(row8[k]) * (double)S[n] * bf16_to_double(xr8[k]);",
                         "e4m3_to_double(row8[k]) * bf16_to_double(xr8[k]);"),
    "fp8_scale_row_0": ("e4m3_to_double(row8[k]) * (double)S[n] * bf16_to_double(xr8[k]);",
                        "e4m3_to_double(row8[k]) * (double)S[0] * bf16_to_double(xr8[k]);"),
    "fp8_row_stride_K": ("const uint8_t *row8 = Wq + n * ldq;", "const uint8_t *row8 = Wq + n * K;"),
    "fp8_nan_not_nan": ("if (e8 == 0xF && m8 == 0x7) return NAN;", "if (e8 == 0xF && m8 == 0x7) return 480.0;"),
}


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant_src = tmp_path / f"mutant_{name}.c"
    mutant_src.write_text(src.replace(old, new))
    so = oracle.build(str(mutant_src), str(tmp_path / f"libmutant_{name}.so"), force=True)
    lib = oracle.OracleLib(so)
    fails = oracle_pins.failures(lib)
    assert fails, f"planted mistake {name} passed every pin"


def test_accept_rule():
    y_ref = np.array([[1.0, -2.0, 0.0, 3.0]])
    scale = np.array([[10.0, 10.0, 0.0, 1.0]])
    y_gpu = np.array([[1.0 + 9e-5, -2.0 - 1.1e-4, -0.0, np.nan]])
    ok = oracle.accept(y_gpu, y_ref, scale, rtol=1e-5)
    assert ok.tolist() == [[True, False, True, False]]


def test_threads_do_not_change_results(oracle_lib):
    from memory_bound_decode_gb300 import inputs
    W = inputs.bits(inputs.weight(257, 513, seed=1))
    x = inputs.bits(inputs.activations(2, 513, seed=1))
    y1, s1 = oracle_lib.gemv(W, x, threads=1)
    y4, s4 = oracle_lib.gemv(W, x, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(s1, s4)


def test_argument_checks(oracle_lib):
    W = np.zeros((4, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle_lib.gemv(W, np.zeros((1, 9), dtype=np.uint16))
    with pytest.raises(TypeError):
        oracle_lib.gemv(W.astype(np.int32), np.zeros((1, 8), dtype=np.uint16))
    with pytest.raises(ValueError):
        oracle_lib.gemv_one(W, np.zeros((1, 8), dtype=np.uint16), 1, 0)


def test_source_is_test_infrastructure():
    head = open(oracle.SOURCE).read(600)
    assert "TEST INFRASTRUCTURE ONLY" in head
    assert os.path.basename(oracle.SOURCE) == "gemv_oracle.c"
