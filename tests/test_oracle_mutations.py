"""The oracle's pins must catch plausible mistakes (CPU only).

Each case copies the oracle source, plants one mistake in the copy, builds it
with gcc into a temporary directory and runs the pin suite against it; at least
one pin must fail.  The committed oracle is never modified.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_codecs as codecs
from tests import test_oracle_dgrad as dgrad
from tests import test_oracle_gemm as gemm
from tests import test_oracle_lora_grads as lgrads
from tests import test_oracle_quantize as quant

SRC = os.path.join(os.path.dirname(oracle.__file__), "nvfp4_oracle.c")

# (name, text to find, replacement)
MUTATIONS = [
    ("tensor scale constant", "a / 2688.0f", "a / 2560.0f"),
    ("nibble order", "if ((k & 1) == 0)\n                *byte", "if ((k & 1) == 1)\n                *byte"),
    ("ties away from even", "(d == bd && (c & 1) == 0)", "(d == bd && (c & 1) == 1)"),
    ("E2M1 exponent bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("E4M3 subnormal exponent", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("E4M3 mantissa width", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 16.0, e - 7)"),
    ("no saturation", "if (!(x_abs < grid[n - 1]))\n        return n - 1;", ""),
    ("block amax without abs", "float v = fabsf(orc_bf16_to_f32(row[b * 16 + i]));",
     "float v = orc_bf16_to_f32(row[b * 16 + i]);"),
    ("block scale from 4 instead of 6", "float d = 6.0f * c->s_t;", "float d = 4.0f * c->s_t;"),
    ("sign of code dropped", "return (signbit(x) ? 8 : 0) | mag;", "return mag;"),
    ("noise ignored", "float p = orc_bf16_to_f32(b) * z[k];", "float p = orc_bf16_to_f32(b);"),
    ("noisy input not rounded to bf16", "b = orc_f32_to_bf16(p);",
     "b = orc_f32_to_bf16(orc_bf16_to_f32(b) * (1.0f + (z[k] - 1.0f) * 0.5f));"),
    ("LoRA scale dropped", "c->y[m * c->N + n] = acc + c->s * lora;", "c->y[m * c->N + n] = acc + lora;"),
    ("LoRA B transposed", "c->B[n * c->r + j]", "c->B[j * c->N + n]"),
    ("wrong block index in GEMM",
     "c->scales[n * (c->K / 16) + k / 16]) * c->s_t;\n            acc += (double)orc_bf16_to_f32(c->xp",
     "c->scales[n * (c->K / 16) + k / 32]) * c->s_t;\n            acc += (double)orc_bf16_to_f32(c->xp"),
    ("tensor scale dropped in GEMM", "* c->s_t;\n            acc += (double)orc_bf16_to_f32(c->xp",
     ";\n            acc += (double)orc_bf16_to_f32(c->xp"),
    ("dequant drops tensor scale", "float v = vd * s_t;", "float v = vd;"),
    ("scale update divides wrong way", "p / s_t;", "p * s_t;"),
    ("reciprocal instead of division", "float x = orc_bf16_to_f32(row[b * 16 + i]) / S_b;",
     "float x = orc_bf16_to_f32(row[b * 16 + i]) * (1.0f / S_b);"),
    ("zero block scale not special-cased", "if (S_b != 0.0f) {", "if (1) {"),
    ("tensor amax without abs", "float v = fabsf(orc_bf16_to_f32(w[i]));", "float v = orc_bf16_to_f32(w[i]);"),
    ("LoRA branch without noise",
     "t += (double)orc_bf16_to_f32(xp[m * K + k]) * (double)orc_bf16_to_f32(A[j * K + k]);\n            T[m * r + j] = t;",
     "t += (double)orc_bf16_to_f32(x[m * K + k]) * (double)orc_bf16_to_f32(A[j * K + k]);\n            T[m * r + j] = t;"),
    ("frozen scale ignored", "    if (given) {\n        s_t = *st_io;", "    if (0) {\n        s_t = *st_io;"),
    ("dequant scales by s_t before the block scale",
     "float vd = (float)(orc_e2m1_value(code_at(codes, K, n, k)) *\n                               orc_e4m3_value(scales[n * (K / 16) + k / 16]));\n            float v = vd * s_t;",
     "float vd = (float)orc_e2m1_value(code_at(codes, K, n, k)) * s_t;\n            float v = vd * (float)orc_e4m3_value(scales[n * (K / 16) + k / 16]);"),
    ("LoRA term subtracted", "c->y[m * c->N + n] = acc + c->s * lora;", "c->y[m * c->N + n] = acc - c->s * lora;"),
    ("GEMM accumulates in float", "        double acc = 0.0;\n        for (int64_t k = 0; k < c->K; k++) {",
     "        float acc = 0.0f;\n        for (int64_t k = 0; k < c->K; k++) {"),
    ("LoRA down-projection in float", "            double t = 0.0;", "            float t = 0.0f;"),
    ("negative scale parameter not zeroed", "(s_t == 0.0f || p <= 0.0f) ? 0.0f : p / s_t",
     "(s_t == 0.0f) ? 0.0f : fabsf(p) / s_t"),
    ("LoRA A read transposed",
     "(double)orc_bf16_to_f32(A[j * K + k]);\n            T[m * r + j] = t;",
     "(double)orc_bf16_to_f32(A[k * r + j]);\n            T[m * r + j] = t;"),
    ("block amax over half the block", "        float a_b = 0.0f;\n        for (int i = 0; i < 16; i++) {",
     "        float a_b = 0.0f;\n        for (int i = 0; i < 8; i++) {"),
    ("LoRA scale on the base term", "c->y[m * c->N + n] = acc + c->s * lora;", "c->y[m * c->N + n] = c->s * acc + lora;"),
    ("output rows and columns swapped", "c->y[m * c->N + n] = acc + c->s * lora;",
     "c->y[n * c->M + m] = acc + c->s * lora;"),
    ("array encoder drops the short last piece", "for_rows((n + c.per - 1) / c.per, nthreads, enc_row, &c);",
     "for_rows(n / c.per, nthreads, enc_row, &c);"),
    ("array encoder swaps the two encoders",
     "c->out[i] = (uint8_t)(c->which == 0 ? orc_e2m1_encode(c->x[i]) : orc_e4m3_encode_nonneg(c->x[i]));",
     "c->out[i] = (uint8_t)(c->which == 1 ? orc_e2m1_encode(c->x[i]) : orc_e4m3_encode_nonneg(c->x[i]));"),
    ("dgrad noise dropped", "c->dx[m * c->K + k] = c->z ? g * (double)c->z[k] : g;",
     "c->dx[m * c->K + k] = g;"),
    ("dgrad LoRA scale dropped", "double g = acc + c->s * lora;", "double g = acc + lora;"),
    ("dgrad LoRA term subtracted", "double g = acc + c->s * lora;", "double g = acc - c->s * lora;"),
    ("dgrad LoRA B read transposed", "(double)orc_bf16_to_f32(B[n * r + j]);\n            U[m * r + j] = u;",
     "(double)orc_bf16_to_f32(B[j * N + n]);\n            U[m * r + j] = u;"),
    ("dgrad LoRA A read transposed", "(double)orc_bf16_to_f32(c->A[j * c->K + k])",
     "(double)orc_bf16_to_f32(c->A[k * c->r + j])"),
    ("dgrad tensor scale dropped", "* c->s_t;\n            acc += (double)orc_bf16_to_f32(c->dy",
     ";\n            acc += (double)orc_bf16_to_f32(c->dy"),
    ("dgrad block index from the wrong column",
     "c->scales[n * (c->K / 16) + k / 16]) * c->s_t;\n            acc += (double)orc_bf16_to_f32(c->dy",
     "c->scales[n * (c->K / 16) + k / 32]) * c->s_t;\n            acc += (double)orc_bf16_to_f32(c->dy"),
    ("dgrad LoRA down-projection in float", "            double u = 0.0;", "            float u = 0.0f;"),
    ("dgrad uses the first dY row for every row", "acc += (double)orc_bf16_to_f32(c->dy[m * c->N + n]) * d;",
     "acc += (double)orc_bf16_to_f32(c->dy[n]) * d;"),
    ("dB scale dropped", "c->db[n * c->r + j] = c->s * acc;", "c->db[n * c->r + j] = acc;"),
    ("dA scale dropped", "c->da[j * c->K + k] = c->s * acc;", "c->da[j * c->K + k] = acc;"),
    ("dB from U instead of T", "* c->T[m * c->r + j];", "* c->U[m * c->r + j];"),
    ("dA from T instead of U", "acc += c->U[m * c->r + j] * (double)orc_bf16_to_f32(c->xp",
     "acc += c->T[m * c->r + j] * (double)orc_bf16_to_f32(c->xp"),
    ("dB written transposed", "c->db[n * c->r + j] = c->s * acc;", "c->db[j * c->N + n] = c->s * acc;"),
    ("LoRA gradients without noise",
     "    orc_noisy_input(x, z, M, K, xp);\n    for (int64_t m = 0; m < M; m++)\n        for (int64_t j = 0; j < r; j++) {\n            double t = 0.0, u = 0.0;",
     "    orc_noisy_input(x, NULL, M, K, xp);\n    for (int64_t m = 0; m < M; m++)\n        for (int64_t j = 0; j < r; j++) {\n            double t = 0.0, u = 0.0;"),
    ("U with B read transposed", "(double)orc_bf16_to_f32(B[n * r + j]);\n            T[m * r + j] = t;",
     "(double)orc_bf16_to_f32(B[j * N + n]);\n            T[m * r + j] = t;"),
    ("T of the gradients with A read transposed",
     "(double)orc_bf16_to_f32(A[j * K + k]);\n            for (int64_t n = 0; n < N; n++)",
     "(double)orc_bf16_to_f32(A[k * r + j]);\n            for (int64_t n = 0; n < N; n++)"),
    ("array encoder skips the last element of each piece",
     "int64_t lo = r * c->per, hi = lo + c->per < c->n ? lo + c->per : c->n;",
     "int64_t lo = r * c->per, hi = lo + c->per - 1 < c->n ? lo + c->per - 1 : c->n;"),
]

PINS = [
    codecs.test_e2m1_grid_matches_golden,
    codecs.test_e2m1_ties_match_golden,
    codecs.test_e2m1_encoder_vs_thresholds,
    codecs.test_e4m3_decode_all_bytes_vs_torch,
    codecs.test_e4m3_encoder_vs_torch_in_range,
    codecs.test_e4m3_encoder_saturates,
    lambda o: codecs.test_encode_array_matches_independent_encoders(o, 5),
    quant.test_worked_example,
    lambda o: quant.test_grid_round_trip(o, False),
    lambda o: quant.test_grid_round_trip(o, True),
    lambda o: quant.test_error_bound(o, "normal_outliers"),
    lambda o: quant.test_error_bound(o, "student_t"),
    quant.test_subnormal_scale_blocks_saturate,
    quant.test_exact_ties_resolve_to_even_code_at_every_scale,
    quant.test_scale_only_update_merge_is_bit_identical,
    quant.test_round_scales_edge_values,
    quant.test_sign_symmetry,
    quant.test_frozen_scale_used_verbatim,
    lambda o: gemm.test_gemm_vs_exact_rationals(o, 3, 5, 32, 2),
    lambda o: gemm.test_gemm_vs_exact_rationals(o, 2, 8, 48, 4),
    gemm.test_gemm_dyadic_is_exact,
    gemm.test_power_of_two_noise_equals_prescaled_input_and_scaled_weight,
    gemm.test_degenerate_cases,
    lambda o: dgrad.test_adjoint_identity_exact(o, 3, 16, 64, 4),
    lambda o: dgrad.test_adjoint_identity_exact(o, 5, 40, 128, 8),
    lambda o: dgrad.test_matches_float64_autograd(o, True, True),
    lambda o: dgrad.test_vs_exact_rationals(o, 2, 6, 32, 3),
    dgrad.test_degenerate_cases,
    lambda o: lgrads.test_linear_in_each_factor_exact(o, 3, 16, 64, 4),
    lambda o: lgrads.test_matches_float64_autograd(o, True),
    lgrads.test_vs_exact_rationals,
    lgrads.test_degenerate_cases,
]


def _build_mutant(text, tmp):
    path = os.path.join(tmp, "mutant.c")
    with open(path, "w") as f:
        f.write(text)
    so = os.path.join(tmp, "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", path, "-o", so, "-lm"])
    return so


def _first_failing_pin():
    for pin in PINS:
        try:
            pin(oracle)
        except (AssertionError, ValueError):
            return pin
    return None


def test_unmutated_copy_passes_every_pin():
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(open(SRC).read(), tmp)
        prev = oracle.use_library(so)
        try:
            assert _first_failing_pin() is None
        finally:
            oracle.use_library(None)


@pytest.mark.parametrize("name,find,repl", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, find, repl):
    src = open(SRC).read()
    assert src.count(find) == 1, f"mutation site for '{name}' not unique"
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(src.replace(find, repl), tmp)
        oracle.use_library(so)
        try:
            assert _first_failing_pin() is not None, f"no pin catches: {name}"
        finally:
            oracle.use_library(None)
