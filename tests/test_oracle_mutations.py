"""The oracle's pins bite: plant one plausible slip at a time in a temporary
copy of the oracle's C source (CPU only), rebuild it, and check that a pin in
test_oracle_pins fails against that build."""
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild

import test_oracle_pins as pins

MUTATIONS = [
    ("scale divides by 128", "float s = amax / 127.0f;", "float s = amax / 128.0f;",
     "test_quant_invariants_and_closed_forms", ()),
    ("ties away from zero", "float r = rintf(t);", "float r = roundf(t);",
     "test_quant_matches_torch_round_half_even", ()),
    ("exp drops the low part of ln 2", "r = fmaf(-n, ln2_lo, r);", "r = r + 0.0f;",
     "test_exp_spec_accuracy_and_special_values", ()),
    ("exp cubic coefficient off", "const float c3 = 1.66666671633720397949218750000000e-1f;",
     "const float c3 = 1.6660e-1f;", "test_exp_spec_accuracy_and_special_values", ()),
    ("sigmoid sign", "float e = oracle_exp_f32(-g);", "float e = oracle_exp_f32(g);",
     "test_swiglu_against_float64_and_closed_forms", ()),
    ("gate and up swapped", "float g = oracle_bf16_to_f32(y13[r * 2 * I + j]);",
     "float g = oracle_bf16_to_f32(y13[r * 2 * I + I + j]);", "test_swiglu_gate_is_first_half", ()),
    ("bias from the wrong column", "t = t + oracle_bf16_to_f32(bias[n]);",
     "t = t + oracle_bf16_to_f32(bias[0]);", "test_epilogue_against_float64", ()),
    ("weight read transposed", "for (int64_t k = 0; k < K; ++k) a += (int32_t)qr[k] * (int32_t)wr[k];\n      acc[m * N + n] = a;",
     "for (int64_t k = 0; k < K; ++k) a += (int32_t)qr[k] * (int32_t)w[k * N + n];\n      acc[m * N + n] = a;",
     "test_gemm_acc_matches_int64_matmul", (7, 96, 13)),
    ("grouped row scale indexed inside the group", "y[r * N + n] = epilogue_one(a, x_scale[r], se[n], NULL, n);",
     "y[r * N + n] = epilogue_one(a, x_scale[r - off], se[n], NULL, n);",
     "test_grouped_golden_example_against_numpy", ()),
    ("group-list sum not checked", "return total == R ? ORC_OK : ORC_ERR_GROUP_LIST;", "return ORC_OK;",
     "test_grouped_rejects_bad_group_lists", ()),
    ("pre-quantised input quantised again", "if (x_scale == NULL) {", "if (1) {",
     "test_moe_chain_composition_and_no_double_quant", ()),
    ("routed row not advanced", "        pos[i] = (int32_t)row;\n        ++row;", "        pos[i] = (int32_t)row;",
     "test_route_is_a_stable_sort_by_expert", (50, 4, 9, True)),
    ("expert id upper bound off by one", "topk_ids[i] >= E) return ORC_ERR_TOPK_IDS;",
     "topk_ids[i] > E) return ORC_ERR_TOPK_IDS;", "test_route_rejects_ids_outside_the_experts", ()),
    ("routed scale taken from the wrong token", "xs[r] = st[t];", "xs[r] = st[(t + 1) % T];",
     "test_permute_quant_is_quant_of_the_gathered_rows", (True,)),
    ("combine drops the last choice", "for (int64_t j = 0; j < k; ++j) {\n        const float v",
     "for (int64_t j = 0; j + 1 < k; ++j) {\n        const float v", "test_combine_against_float64", ()),
    ("weight channel read from the first expert", "oracle_dynamic_quant(w + row * K, 1, K, q + row * K, scale + row);",
     "oracle_dynamic_quant(w + n * K, 1, K, q + row * K, scale + row);", "test_weight_quant_is_per_output_channel", ()),
    ("static correction added instead of subtracted", "const float t = rintf(a - c);", "const float t = rintf(a + c);",
     "test_static_path_approximates_the_float_layer", (9,)),
    ("static offset added before rounding", "double c = (double)rintf(t) + (double)o;",
     "double c = (double)rintf(t + (float)o);", "test_static_quant_brute_force_and_closed_forms", ()),
    ("static codes clamped at -127", "if (c < -128.0) c = -128.0;", "if (c < -127.0) c = -127.0;",
     "test_static_quant_brute_force_and_closed_forms", ()),
    ("MX shared exponent one too high", "shared = (e - 1) - 8;", "shared = e - 8;",
     "test_mx_quant_closed_forms_and_bounds", ()),
    ("E4M3 without saturation", "if (a >= 448.0) return sign | 0x7E;", "if (a >= 464.0) return sign | 0x7F;",
     "test_e4m3_encode_decode_against_torch", ()),
    ("MX matmul drops the weight scale", "acc += part * pow2d((int)sa[m * G + g] - 127) * pow2d((int)sw[n * G + g] - 127);",
     "acc += part * pow2d((int)sa[m * G + g] - 127);", "test_mx_matmul_against_float64", ()),
    ("combine sums in double", "      float s = 0.0f;\n      for (int64_t j", "      double s = 0.0;\n      for (int64_t j",
     "test_combine_closed_forms_and_order", ()),
]


@pytest.mark.parametrize("name,old,new,pin,args", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_slip_is_caught(tmp_path, name, old, new, pin, args):
    src = open(obuild.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(mutated)
    so_path = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", *obuild.CFLAGS, str(c_path), "-o", so_path, "-lm"], check=True,
                   capture_output=True)
    prev = oracle.use_library(so_path)
    try:
        with pytest.raises((AssertionError, oracle.OracleError)):
            getattr(pins, pin)(*args)
    finally:
        oracle.restore_library(prev)
