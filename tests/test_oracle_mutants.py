"""The pins are strong enough to catch plausible mistakes: each mistake below is
planted in a copy of oracle.c (on the CPU, in a temporary directory), the copy is
built and swapped in for the oracle, and at least one pin must then fail.  The
unmodified oracle passes the same pins (the first case)."""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_dispatch as pd
import test_oracle_ffn_combine as pf
import test_oracle_mxfp8 as pm
import test_oracle_route as pr

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# name -> (text in oracle.c, planted replacement)
MUTANTS = {
    "none": None,
    "ties_to_higher_id": ("if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] >= l[best]) best = e;"),
    "weights_not_renormalised": ("w[j] = exp((double)l[idx[j]] - m) / s;", "w[j] = exp((double)l[idx[j]] - m);"),
    "silu_sign": ("double silu = g / (1.0 + exp(-g));", "double silu = g / (1.0 + exp(g));"),
    "gate_and_up_swapped": ("double silu = g / (1.0 + exp(-g));\n        act[i] = silu * u;",
                            "double silu = u / (1.0 + exp(-u));\n        act[i] = silu * g;"),
    "down_weights_transposed": ("acc += bf16_widen(rd[i]) * act[i];",
                                "acc += bf16_widen(wd[(int64_t)i * H + h]) * act[i];"),
    "dispatch_rows_descending": ("int32_t r = offsets[e - e0] + fill[e - e0]++;",
                                 "int32_t r = offsets[e - e0 + 1] - 1 - fill[e - e0]++;"),
    "combine_ignores_weights": ("o[h] += w * (double)y_perm[(int64_t)r * H + h];",
                                "o[h] += (double)y_perm[(int64_t)r * H + h];"),
    "layer_ignores_weights": ("for (int h = 0; h < H; ++h) o[h] += w[j] * y[h];",
                              "for (int h = 0; h < H; ++h) o[h] += y[h];"),
    "mx_scale_off_by_one": ("int c = p - 8 + 127;", "int c = p - 7 + 127;"),
    "mx_saturates_to_nan_code": ("if (a >= 448.0) return sign | 0x7e; /* saturate (also the rounding of 448..464) */",
                                 "if (a >= 448.0) return sign | 0x7f;"),
    "mx_round_half_away": ("double m = nearbyint(a / q);", "double m = floor(a / q + 0.5);"),
    "mx_h_not_quantised": ("mx_dequantize_row(I, hq, hs, hd);", "memcpy(hd, h, sizeof(double) * (size_t)I);"),
    # (memory-safe mistakes only: a planted out-of-bounds index could take the test process down)
    "up_uses_gate_weights": ("for (int h = 0; h < H; ++h) u += bf16_widen(ru[h]) * x[h];",
                             "for (int h = 0; h < H; ++h) u += bf16_widen(rg[h]) * x[h];"),
    "combine_first_slot_weight_for_all": ("double w = (double)topk_w[t * k + j];", "double w = (double)topk_w[t * k];"),
    "layer_skips_first_local_expert": ("if (e < e0 || e >= e1) continue;", "if (e <= e0 || e >= e1) continue;"),
    "grouped_row_expert_boundaries_shifted": ("if (r >= offsets[q] && r < offsets[q + 1]) { e = q; break; }",
                                              "if (r > offsets[q] && r <= offsets[q + 1]) { e = q; break; }"),
    "mx_amax_without_abs": ("for (int i = 0; i < len; ++i) amax = fmax(amax, fabs(v[i]));",
                            "for (int i = 0; i < len; ++i) amax = fmax(amax, v[i]);"),
    "e4m3_subnormal_step_halved": ("        q = ldexp(1.0, -9);", "        q = ldexp(1.0, -10);"),
    "nonfinite_logits_not_detected": ("        if (!isfinite(l[e])) return ORACLE_ERR_NONFINITE;", "        (void)0;"),
    "softmax_over_all_experts": ("for (int j = 0; j < k; ++j) s += exp((double)l[idx[j]] - m);",
                                 "for (int j = 0; j < E; ++j) s += exp((double)l[j] - m);"),
    "nonlocal_pair_row_zero": ("            pair_row[p] = -1;", "            pair_row[p] = 0;"),
    "activation_without_up": ("        act[i] = silu * u;", "        act[i] = silu;"),
    "layer_x_of_first_token": ("for (int h = 0; h < H; ++h) xd[h] = bf16_widen(x[t * H + h]);",
                               "for (int h = 0; h < H; ++h) xd[h] = bf16_widen(x[h]);"),
    "layer_first_slot_weight": ("for (int h = 0; h < H; ++h) o[h] += w[j] * y[h];",
                                "for (int h = 0; h < H; ++h) o[h] += w[0] * y[h];"),
    "layer_first_expert_weights": ("swiglu_ffn(H, I, xd, w_gate + (int64_t)el * I * H, w_up + (int64_t)el * I * H,",
                                   "swiglu_ffn(H, I, xd, w_gate, w_up,"),
    "mx_ffn_up_from_gate_weights": ("mx_dequantize_row(H, wuq + wr * H, wus + wr * (H / 32), w);",
                                    "mx_dequantize_row(H, wgq + wr * H, wgs + wr * (H / 32), w);"),
    "mx_ffn_silu_sign": ("h[i] = g / (1.0 + exp(-g)) * u;", "h[i] = g / (1.0 + exp(g)) * u;"),
    "mx_ffn_gate_up_rows_of_expert_0": ("const int64_t wr = (int64_t)e * I + i;", "const int64_t wr = i;"),
    "mx_ffn_down_rows_of_expert_0": ("const int64_t wr = (int64_t)e * H + j;", "const int64_t wr = j;"),
    "mx_dequantise_scale_bias_126": ("out[k] = e4m3_decode(q[k]) * ldexp(1.0, (int)s[k / 32] - 127);",
                                     "out[k] = e4m3_decode(q[k]) * ldexp(1.0, (int)s[k / 32] - 126);"),
}

PINS = [
    lambda: pr.test_selection_matches_full_sort(16, 4),
    lambda: pr.test_signed_zero_ties_to_lower_id(),
    lambda: pr.test_hand_worked_example(),
    lambda: pr.test_two_expert_closed_form(),
    lambda: pr.test_weights_equal_renormalised_full_softmax(),
    lambda: pr.test_nonfinite_logit_is_an_error(float("nan")),
    lambda: pd.test_dispatch_invariants(16, 4, 3, 11),
    lambda: pf.test_single_expert_is_textbook_mlp(),
    lambda: pf.test_identity_weights_closed_form(),
    lambda: pf.test_dense_masked_formula(0, 6),
    lambda: pf.test_grouped_rows_match_textbook(),
    lambda: pf.test_combine_is_slot_ordered_weighted_gather(),
    lambda: pm.test_e4m3_table_values(),
    lambda: pm.test_nearest_code_by_exhaustive_search(),
    lambda: pm.test_subnormal_codes_by_exhaustive_search(),
    lambda: pm.test_scale_code_closed_form(),
    lambda: pm.test_scale_follows_largest_magnitude_of_either_sign(),
    lambda: pm.test_ties_signed_zero_and_saturation(),
    lambda: pm.test_mx_ffn_against_dequantised_float64(64, 32, 2),
    lambda: pm.test_mx_ffn_near_bf16_oracle_when_operands_are_exact(),
]


def build_variant(tmp_path, name):
    src = open(SRC).read()
    if MUTANTS[name] is not None:
        old, new = MUTANTS[name]
        assert src.count(old) == 1, f"mutation site of {name} not found once in oracle.c"
        src = src.replace(old, new)
    c = tmp_path / f"oracle_{name}.c"
    so = tmp_path / f"liboracle_{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", str(c), "-o", str(so), "-lm"], check=True)
    return oracle._bind(ctypes.CDLL(str(so)))


def failing_pins(lib):
    saved = oracle._load()
    oracle._lib = lib
    failed = 0
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed += 1
    finally:
        oracle._lib = saved
    return failed


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    failed = failing_pins(build_variant(tmp_path, name))
    if name == "none":
        assert failed == 0
    else:
        assert failed >= 1, f"no pin caught the planted mistake {name}"
