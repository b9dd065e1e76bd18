"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Every mutant is the oracle's C source with one snippet replaced, compiled with
the oracle's own flags into a temporary folder and loaded as a separate library.
The test passes when at least one pin of ``tests/pins.py`` fails on every mutant,
and every snippet still occurs exactly once in the real source (so a stale
mutation cannot pass silently).  No GPU is involved.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import pins

MUTANTS = {
    # rounding
    "ties_away_from_even": ("idx = (lo % 2 == 0) ? lo : hi;", "idx = hi;"),
    "sign_dropped": ("return (uint8_t)((neg << sign_shift) | idx);", "return (uint8_t)(idx);"),
    "no_saturation_to_max": ("    if (a >= mag[n - 1]) {\n        idx = n - 1;",
                             "    if (a >= mag[n - 1]) {\n        idx = n - 2;"),
    "e4m3_wrong_bias": ("mag = ldexp(1.0 + man / 8.0, exp - 7);", "mag = ldexp(1.0 + man / 8.0, exp - 8);"),
    # NVFP4 per-token scale
    "scale_constant_2048": ("float s_t = amax / 2688.0f;", "float s_t = amax / 2048.0f;"),
    "block_divisor_without_6": ("float d = 6.0f * s_t;", "float d = s_t;"),
    "reciprocal_multiply": ("float q = bf16_value(xb[j]) / e;", "float q = bf16_value(xb[j]) * (1.0f / e);"),
    "row_amax_from_first_block": (
        "        for (int64_t j = 0; j < k; ++j) {\n            float a = fabsf(bf16_value(xr[j]));",
        "        for (int64_t j = 0; j < 16; ++j) {\n            float a = fabsf(bf16_value(xr[j]));"),
    "block_amax_half_block": (
        "            for (int j = 0; j < 16; ++j) {\n                float a = fabsf(bf16_value(xb[j]));",
        "            for (int j = 0; j < 8; ++j) {\n                float a = fabsf(bf16_value(xb[j]));"),
    "nibbles_swapped": ("if (kk % 2 == 0)", "if (kk % 2 == 1)"),
    "zero_scale_block_divided": ("            if (sb_val == 0.0)\n                continue; /* block codes stay 0x0 */\n",
                                 ""),
    "dequant_drops_token_scale": ("out[t * k + j] = fme_orc_e2m1_value(c) * sb * (double)scale[t];",
                                  "out[t * k + j] = fme_orc_e2m1_value(c) * sb;"),
    # MXFP8
    "mx_emax_7": ("int code = u - 8 + 127;", "int code = u - 7 + 127;"),
    "mx_zero_block_scale_127": ("    if (amax == 0.0f)\n        return 0;", "    if (amax == 0.0f)\n        return 127;"),
    "mx_element_scale_off_by_one": ("double q = ldexp((double)v[j], 127 - (int)sc);",
                                    "double q = ldexp((double)v[j], 128 - (int)sc);"),
    "colwise_pads_to_32": ("int64_t padded = ((n_g + 127) / 128) * 128;", "int64_t padded = ((n_g + 31) / 32) * 32;"),
    # GEMM
    "swiglu_sigmoid_of_minus_g": ("h[t * inter + j] = g / (1.0 + exp(-g)) * u;",
                                  "h[t * inter + j] = g / (1.0 + exp(g)) * u;"),
    "swiglu_gate_up_halves_swapped": ("const double g = (double)bf16_value(row[j]);\n            const double u = (double)bf16_value(row[inter + j]);",
                                      "const double u = (double)bf16_value(row[j]);\n            const double g = (double)bf16_value(row[inter + j]);"),
    "swiglu_drops_up": ("h[t * inter + j] = g / (1.0 + exp(-g)) * u;", "h[t * inter + j] = g / (1.0 + exp(-g));"),
    "swiglu_f64_sigmoid_of_minus_g": ("const double silu = g / (1.0 + exp(-g));",
                                      "const double silu = g / (1.0 + exp(g));"),
    "swiglu_f64_halves_swapped": ("            const double g = row[j];\n            const double u = row[inter + j];",
                                  "            const double u = row[j];\n            const double g = row[inter + j];"),
    "mx_ceil_ignores_exact_powers": ("const int up = (m == 0.5) ? e2 - 1 : e2;", "const int up = e2;"),
    "mx_ceil_is_floor": ("const int up = (m == 0.5) ? e2 - 1 : e2;", "const int up = e2 - 1;"),
    "mx_ceil_divides_by_256": ("frexp((double)amax / 448.0, &e2);", "frexp((double)amax / 256.0, &e2);"),
    "pertensor_keeps_row_amax": ("        if (per_tensor)\n            amax = tensor_amax;\n", ""),
    "pertensor_amax_of_first_row": ("for (int64_t i = 0; i < rows * k; ++i)", "for (int64_t i = 0; i < k; ++i)"),
    "swiglu_bwd_reads_up_as_gate": ("const double g = (double)bf16_value(y_gu[t * 2 * inter + j]);",
                                    "const double g = (double)bf16_value(y_gu[t * 2 * inter + inter + j]);"),
    "swiglu_bwd_drops_sigma_derivative": ("d * u * (s + g * s * (1.0 - s))", "d * u * s"),
    "swiglu_bwd_one_minus_s_as_s": ("d * u * (s + g * s * (1.0 - s))", "d * u * (s + g * s * s)"),
    "swiglu_bwd_halves_swapped": ("d_gu[t * 2 * inter + j] = d * u", "d_gu[t * 2 * inter + inter + j] = d * u"),
    "swiglu_bwd_du_uses_u": ("d_gu[t * 2 * inter + inter + j] = d * g * s;", "d_gu[t * 2 * inter + inter + j] = d * u * s;"),
    "route_unstable": ("        for (int64_t a = 0; a < n; ++a) {\n            if (ids[a] == e) {",
                       "        for (int64_t a = n - 1; a >= 0; --a) {\n            if (ids[a] == e) {"),
    "route_offsets_not_summed": ("offsets[e + 1] += offsets[e];", "offsets[e + 1] += 0;"),
    "route_invalid_kept_as_last": ("            row_of[a] = -1;", "            row_of[a] = n - 1;"),
    "combine_fp64_sum": ("            float acc = 0.0f;\n", "            double acc = 0.0;\n"),
    "combine_reversed_k": ("for (int32_t k = 0; k < top_k; ++k) {\n                const int32_t r",
                           "for (int32_t k = top_k - 1; k >= 0; --k) {\n                const int32_t r"),
    "combine_fused_multiply_add": ("                acc = acc + prod;",
                                   "                acc = fmaf(w[t * top_k + k], bf16_value(y[(int64_t)r * n + j]), acc);"),
    "combine_ties_away": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))", "if (lower >= 0x8000u)"),
    "combine_truncates": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))", "if (0)"),
    "gemm_transposed_operand": ("acc += a[i * k + q] * b[j * k + q];", "acc += a[i * k + q] * b[q * n + j];"),
    "gemm_drops_last_term": ("for (int64_t q = 0; q < k; ++q)\n                acc +=",
                             "for (int64_t q = 0; q < k - 1; ++q)\n                acc +="),
}


def _run_pins(lib_path):
    orc = oracle.Oracle(lib=oracle.load(lib_path))
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
        except pytest.skip.Exception:
            pass
        except Exception as exc:  # a crash inside a pin also counts as caught
            failed.append(f"{check.__name__}:{type(exc).__name__}")
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation snippet for {name} no longer matches the oracle"
    mutated = tmp_path / f"mutant_{name}.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / f"libmutant_{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib), str(mutated), "-lm"], check=True)
    failed = _run_pins(str(lib))
    assert failed, f"no pin caught the planted mistake {name}"


def test_unmutated_copy_passes(tmp_path):
    lib = tmp_path / "libcopy.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib), oracle.SOURCE, "-lm"], check=True)
    failed = _run_pins(str(lib))
    assert not failed, failed
