"""The pins catch plausible mistakes: each case plants one mistake in a copy of the oracle source
(a dropped term, a wrong sign, index, constant, tie rule or operand order), builds it, and checks
that at least one pin fails against the mutant.  Everything runs on the CPU."""
import subprocess

import pytest

import oracle
from oracle import build as obuild
from nvfp4_block_scaled_row_gb300 import synth

import test_oracle_formats as F
import test_oracle_fp16_selector as H
import test_oracle_guided as T
import test_oracle_method as M
import test_oracle_residual as R

SOURCE = open(obuild.SOURCE).read()

# (name, text to replace, replacement)
MUTATIONS = [
    ("e2m1 ties to odd", "(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    ("e2m1 no saturation", "  if (mag > 6.0) mag = 6.0; /* saturate first", "  if (0) mag = 6.0; /* saturate first"),
    ("e4m3 ties to odd", "(err == best_err && (b & 1) == 0)", "(err == best_err && (b & 1) == 1)"),
    ("M = 448 in 4/6", "return mode == ORACLE_MODE_SIX ? 448.0f : 256.0f;", "return 448.0f;"),
    ("c4 = M/a", "out[2] = clamp_to_finite((1.5f * M) / a);", "out[2] = clamp_to_finite(M / a);"),
    ("S_dec = 1/S_enc", "out[3] = a / (6.0f * M);", "out[3] = 1.0f / out[0];"),
    ("ties go to 4", "pick4 = e4 < e6; /* ties go to 6 */", "pick4 = e4 <= e6; /* ties go to 6 */"),
    ("residual sign", "d[i] = fmaf(-r, s, z);", "d[i] = fmaf(r, s, z);"),
    ("error chain index", "for (int i = 0; i < ORACLE_BLOCK; ++i) e = fmaf(d[i], d[i], e);",
     "for (int i = 0; i < ORACLE_BLOCK; ++i) e = fmaf(d[i], d[i ^ 1], e);"),
    ("error chain descending", "for (int i = 0; i < ORACLE_BLOCK; ++i) e = fmaf(d[i], d[i], e);",
     "for (int i = ORACLE_BLOCK - 1; i >= 0; --i) e = fmaf(d[i], d[i], e);"),
    ("error chain in two halves", "for (int i = 0; i < ORACLE_BLOCK; ++i) e = fmaf(d[i], d[i], e);",
     "float h1 = 0.0f; for (int i = 0; i < 8; ++i) { e = fmaf(d[i], d[i], e); "
     "h1 = fmaf(d[8 + i], d[8 + i], h1); } e = e + h1;"),
    ("error chain four interleaved", "for (int i = 0; i < ORACLE_BLOCK; ++i) e = fmaf(d[i], d[i], e);",
     "float E[4] = {0.0f, 0.0f, 0.0f, 0.0f}; for (int i = 0; i < ORACLE_BLOCK; ++i) "
     "E[(i >> 3) * 2 + (i & 1)] = fmaf(d[i], d[i], E[(i >> 3) * 2 + (i & 1)]); "
     "e = (E[0] + E[1]) + (E[2] + E[3]);"),
    ("nibble order", "packed[j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));",
     "packed[j] = (uint8_t)(c[2 * j + 1] | (c[2 * j] << 4));"),
    ("block amax over 8", "for (int i = 0; i < ORACLE_BLOCK; ++i) m = fmaxf(m, fabsf(x[i]));",
     "for (int i = 0; i < ORACLE_BLOCK / 2; ++i) m = fmaxf(m, fabsf(x[i]));"),
    ("dequant drops S_dec", "y[r * cols + k] = oracle_bf16_encode(qs * S_dec);",
     "y[r * cols + k] = oracle_bf16_encode(qs);"),
    ("target not scaled", "float t = z * inv;        /* scaled down", "float t = z;        /* scaled down"),
    ("bf16 ties to odd", "return (uint16_t)((((lo >> 16) & 1u) != 0) ? (hi >> 16) : (lo >> 16));",
     "return (uint16_t)((((lo >> 16) & 1u) == 0) ? (hi >> 16) : (lo >> 16));"),
    ("residual not rounded to bf16",
     "dx[k] = oracle_bf16_encode(oracle_bf16_to_f32(xr[k]) - oracle_bf16_to_f32(y[k]));",
     "dx[k] = (uint16_t)(oracle_bf16_encode(oracle_bf16_to_f32(xr[k])) - y[k]);"),
    ("S_enc = M/a", "out[0] = clamp_to_finite((6.0f * M) / a); /* S_enc */",
     "out[0] = clamp_to_finite(M / a); /* S_enc */"),
    ("guided ignores the rollout", "double v = (fabs(hi - rv) < fabs(lo - rv)) ? hi : lo;",
     "double v = (fabs(hi - tc) < fabs(lo - tc)) ? hi : lo;"),
    ("guided takes the farther neighbour", "double v = (fabs(hi - rv) < fabs(lo - rv)) ? hi : lo;",
     "double v = (fabs(hi - rv) < fabs(lo - rv)) ? lo : hi;"),
    ("fp16 candidate without its scale", "double qs = oracle_e2m1_value(code[i]) * (double)s; /* exact */",
     "double qs = oracle_e2m1_value(code[i]); /* exact */"),
    ("fp16 target not rounded", "double zh = oracle_f16_round((double)z);", "double zh = (double)z;"),
    ("fp16 sum in fp16", "    e = fmaf(d, d, e);\n  }\n  return e;",
     "    e = (float)oracle_f16_round((double)d * d + e);\n  }\n  return e;"),
]


def _small_inputs():
    return [synth.as_u16(synth.generate(0, rows=64)["x"]),
            synth.as_u16(synth.generate(2, rows=12)["x"]),
            synth.as_u16(synth.generate(4, rows=40)["x"])]


def _pins(inputs):
    """The pin checks, run against whatever library oracle._lib currently holds."""
    F.test_e2m1_encode_brute_force()
    F.test_e2m1_ties_go_to_even_mantissa()
    F.test_trace_worked_example()
    F.test_e4m3_encode_matches_torch_in_range()
    F.test_e4m3_encode_saturates_above_range()
    F.test_bf16_encode_matches_torch()
    for mode, m in ((oracle.MODE_FOUR_OVER_SIX, 256.0), (oracle.MODE_SIX, 448.0)):
        F.test_factors_power_of_two_amax_are_exact(mode, m)
    F.test_factors_are_correctly_rounded_quotients(oracle.MODE_FOUR_OVER_SIX, 256)
    M.test_worst_case_error_bounds(inputs, oracle.MODE_FOUR_OVER_SIX)
    M.test_page_example_five_sixths_prefers_four()
    M.test_four_over_six_choice_agrees_with_float64(inputs)
    M.test_ties_go_to_six()
    M.test_block_error_is_one_ascending_chain()
    M.test_per_element_codes_are_nearest(inputs)
    for four in (False, True):
        M.test_idempotent_on_grid_values(four)
    M.test_mode_six_maps_row_max_to_six(inputs)
    M.test_dequant_closed_form(inputs)
    R.test_residual_is_quantize_of_independent_residual(inputs, oracle.MODE_FOUR_OVER_SIX)
    R.test_residual_recovers_most_of_the_error(inputs)
    T.test_trace_worked_example()
    T.test_identity_when_trainer_matches_rollout()
    T.test_choice_is_a_neighbour_and_never_further_than_rtn(1)
    H.test_outputs_differ_only_where_the_choice_flips(inputs)
    H.test_choice_agreement_with_fp32(inputs)
    H.test_fp16_errors_sum_in_fp32_in_element_order()


@pytest.fixture(scope="module")
def inputs():
    return _small_inputs()


def test_pins_pass_on_the_real_oracle(inputs):
    _pins(inputs)


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, old, new, inputs, tmp_path):
    assert SOURCE.count(old) == 1, f"mutation anchor for {name!r} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(SOURCE.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *[f for f in obuild.CFLAGS if f != "-Werror"], str(src), "-o", str(lib),
                    "-lm"], check=True, capture_output=True)
    real = oracle._load()
    try:
        oracle._lib = None
        saved = obuild.build
        obuild.build = lambda force=False: str(lib)
        try:
            oracle._load()
        finally:
            obuild.build = saved
        with pytest.raises((AssertionError, ValueError)):
            _pins(inputs)
    finally:
        oracle._lib = real
