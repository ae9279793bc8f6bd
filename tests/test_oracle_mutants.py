"""The oracle's pins catch plausible mistakes in the oracle.

Each case copies oracle/moe_oracle.c, plants one mistake (a wrong exponent
bias, a swapped nibble, a dropped term, a wrong sign, index or stride, a
transposed operand, an unstable sort, a wrong tie or NaN rule in the routing),
compiles the copy, points the oracle package at it and runs the pins of
tests/test_oracle_pins.py until one fails.
A mutant that passes every pin would be a mistake the pins cannot see.  The
unmutated copy must pass them all.  Every planted index stays inside its array
for the pins' shapes (I <= H, ids inside [0, E) where they index), so a mutant
computes wrong numbers and never reads out of bounds.  CPU only.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_ext as ext
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "moe_oracle.c")

# name -> (text in moe_oracle.c, replacement); each text occurs exactly once
MUTANTS = {
    "e2m1_exponent_bias": ("(int)e - 1)", "(int)e - 2)"),
    "e2m1_subnormal": ("(e == 0) ? 0.5 * (double)m", "(e == 0) ? 1.0 * (double)m"),
    "e2m1_sign_bit": ("s = (code >> 3) & 1u", "s = (code >> 2) & 1u"),
    "e4m3_exponent_bias": ("(int)e - 7)", "(int)e - 6)"),
    "e4m3_subnormal": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_nan_code": ("if (e == 15u && m == 7u)", "if (e == 15u && m == 6u)"),
    "nibble_order": ("(c & 1) ? (byte >> 4) : (byte & 15u)", "(c & 1) ? (byte & 15u) : (byte >> 4)"),
    "scale_block_of_32": ("(size_t)(c / 16)]", "(size_t)(c / 32)]"),
    "scale_row_pitch": ("s[r * (size_t)(K / 16)", "s[r * (size_t)(K / 32)"),
    "packed_row_pitch": ("q[r * (size_t)(K / 2)", "q[r * (size_t)(K / 4)"),
    "tensor_scale_dropped": ("tab_e2m1[nib] * tab_e4m3[sc] * ts;", "tab_e2m1[nib] * tab_e4m3[sc] + 0.0 * ts;"),
    "bf16_shift": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "gate_up_tensor_scales_swapped": ("double tg = (double)gate_ts[e], tu = (double)up_ts[e]",
                                      "double tg = (double)up_ts[e], tu = (double)gate_ts[e]"),
    "gate_reads_up_weights": ("sg += weight_at(gq, gs, tg,", "sg += weight_at(uq, us, tg,"),
    "up_reads_gate_scales": ("su += weight_at(uq, us, tu,", "su += weight_at(uq, gs, tu,"),
    "gate_sum_half_row": ("for (int c = 0; c < H; ++c) {\n            sg +=",
                          "for (int c = 0; c < H / 2; ++c) {\n            sg +="),
    "silu_sign": ("exp(-sg)", "exp(sg)"),
    "silu_on_up": ("hbuf[i] = sg / (1.0 + exp(-sg)) * su;", "hbuf[i] = su / (1.0 + exp(-su)) * sg;"),
    "sigmoid_not_silu": ("hbuf[i] = sg / (1.0 + exp(-sg)) * su;", "hbuf[i] = 1.0 / (1.0 + exp(-sg)) * su;"),
    "down_rows_reversed": ("weight_at(dq, ds, td, I, (size_t)r, i)", "weight_at(dq, ds, td, I, (size_t)(H - 1 - r), i)"),
    "down_sum_not_accumulated": ("acc += weight_at(dq, ds, td, I, (size_t)r, i) * hbuf[i];",
                                 "acc = weight_at(dq, ds, td, I, (size_t)r, i) * hbuf[i];"),
    "down_expert_stride": ("*dq = down_q + (size_t)e * H * (I / 2)", "*dq = down_q + (size_t)e * I * (I / 2)"),
    "x_row_stride": ("x[(size_t)t * H + (size_t)c]", "x[(size_t)t * I + (size_t)c]"),
    "ids_transposed": ("int e = ids[(size_t)t * k + (size_t)j];", "int e = ids[(size_t)j * T + (size_t)t];"),
    "last_slot_dropped": ("for (int j = 0; j < k; ++j) {\n            int e = ids[",
                          "for (int j = 0; j < k - 1; ++j) {\n            int e = ids["),
    "routing_weight_dropped": ("yt[r] += wj * o[r];", "yt[r] += o[r];"),
    "routing_weight_of_slot0": ("w[(size_t)t * k + (size_t)j]", "w[(size_t)t * k]"),
    "bad_id_not_counted": ("++bad;\n                continue;", "continue;"),
    "group_unstable": ("for (int p = 0; p < P; ++p) {\n        int e = ids[p];\n        if (e >= 0 && e < E)",
                       "for (int p = P - 1; p >= 0; --p) {\n        int e = ids[p];\n        if (e >= 0 && e < E)"),
    "group_offsets_not_prefix_sum": ("offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = counts[e];"),
    "group_negative_ids_counted_bad": ("if (e >= E)\n            ++bad;\n        else if (e >= 0)",
                                       "if (e >= E || e < 0)\n            ++bad;\n        else if (e >= 0)"),
    "group_padding_not_minus_one": ("perm[p] = -1;", "perm[p] = 0;"),
    "route_ties_to_larger_index": ("if (best < 0 || v > bv) {", "if (best < 0 || v >= bv) {"),
    "route_nan_compared_as_a_value": ("double v = isnan(lt[e]) ? -INFINITY : (double)lt[e];", "double v = (double)lt[e];"),
    "route_sum_without_max_shift": (": exp(sel[j] - m));", ": exp(sel[j]));"),
    "route_weights_not_normalised": ("(float)(ej / sum)", "(float)(ej)"),
    "route_inf_winner_as_softmax": ("double ej = (m == INFINITY) ? (sel[j] == INFINITY ? 1.0 : 0.0) : exp(sel[j] - m);",
                                    "double ej = exp(sel[j] - m);"),
    "route_ids_of_token_0": ("const float *lt = logits + (size_t)t * E;", "const float *lt = logits;"),
    # the step's extensions: shared expert, expert range, single NVFP4 activation quantisation
    "shared_with_last_slot_weight": ("            for (int r = 0; r < H; ++r)\n                yt[r] += o[r];",
                                     "            for (int r = 0; r < H; ++r)\n                yt[r] += (double)w[(size_t)t * k + (size_t)(k - 1)] * o[r];"),
    "shared_up_scale_for_gate": ("sg_q, sg_s, s_ts + 0,", "sg_q, sg_s, s_ts + 1,"),
    "range_offset_dropped": ("expert_pair_mode(H, I, e - e_lo,", "expert_pair_mode(H, I, e,"),
    "range_outside_counted_bad": ("            if (e < e_lo || e >= e_hi)\n                continue;",
                                  "            if (e < e_lo || e >= e_hi) {\n                ++bad;\n                continue;\n            }"),
    "quant_scale_not_raised": ("        if (tab_e4m3[c] < (double)a && c < 0x7Eu)\n            ++c;",
                               "        if (0)\n            ++c;"),
    "quant_e2m1_ties_up": ("if (d < bd || (d == bd && (c & 1u) == 0))\n            best = c, bd = d;\n    }\n    return best;\n}\n\n/* One row",
                           "if (d <= bd)\n            best = c, bd = d;\n    }\n    return best;\n}\n\n/* One row"),
    "quant_prescale_off_by_one": ("int e = (m <= 1.3125 ? 11 : 10) - E;", "int e = (m <= 1.3125 ? 12 : 10) - E;"),
}


def _pin_checks():
    """The pins, cheapest first, as (name, callable) pairs."""
    small = pins.make_small_case()
    checks = [
        ("e2m1_table", pins.test_e2m1_table_matches_spec),
        ("e4m3_table", pins.test_e4m3_golden_and_library),
        ("dequant_library_route", pins.test_dequant_matches_library_route),
        ("quantizer_roundtrip", pins.test_quantizer_grid_roundtrip_exact),
        ("quantizer_ties", pins.test_quantizer_e2m1_ties_to_even),
        ("group_sorted_16x8", lambda: pins.test_group_against_sorted(16, 8, 256, 1)),
        ("group_sorted_7x4", lambda: pins.test_group_against_sorted(7, 4, 5, 5)),
        ("gate_up_fractions", pins.test_gate_up_exact_against_fractions),
        ("silu_down_torch", pins.test_silu_mul_and_down_against_torch),
        ("dense_mlp", pins.test_dense_mlp_special_case),
        ("combine_torch", pins.test_combine_against_torch),
        ("route_brute_force", lambda: pins.test_route_against_brute_force(16, 256, 8, 1)),
        ("route_ties_nan_extremes", pins.test_route_ties_nan_and_extremes),
        ("route_invariants", pins.test_route_invariants),
        ("quant_row_grid", ext.test_quant_row_is_exact_on_the_grid),
        ("quant_row_ties", ext.test_quant_row_ties_to_even),
        ("quant_row_raised_scale", ext.test_quant_row_raises_the_block_scale),
        ("quant_row_bound", lambda: ext.test_quant_row_scale_sign_invariance_and_bound(0)),
        ("quant_row_zeros", ext.test_quant_row_of_zeros_and_tiny_blocks),
    ]
    ecase = ext.make_case()
    for name in ("shared_expert_alone_is_the_dense_mlp", "shared_expert_adds_after_the_routed_slots",
                 "expert_range_still_flags_ids_past_E", "one_expert_range_is_the_step_with_other_slots_emptied"):
        fn = getattr(ext, "test_" + name)
        checks.append((name, lambda fn=fn: fn(ecase)))
    checks.append(("expert_range_partials", lambda: ext.test_expert_range_partials_sum_to_the_whole_step(ecase, 3)))
    for name in ("zero_weights_give_zero", "token_permutation_permutes_output", "power_of_two_scaling",
                 "slot_linearity", "empty_and_bad_slots", "duplicate_slots_add", "token_subset_matches_full",
                 "thread_count_does_not_change_result"):
        fn = getattr(pins, "test_" + name)
        checks.append((name, lambda fn=fn: fn(small)))
    return checks


def _build(src_text, out_dir, name):
    src = os.path.join(out_dir, name + ".c")
    lib = os.path.join(out_dir, "lib" + name + ".so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-o", lib, src,
                    "-lm"],
                   check=True, capture_output=True)
    return lib


def _first_failing_pin(lib, monkeypatch):
    """Load `lib` as the oracle and return the name of the first pin that fails
    (None if all pass)."""
    monkeypatch.setattr(oracle, "build", lambda force=False: lib)
    monkeypatch.setattr(oracle, "_lib", None)
    for name, check in _pin_checks():
        try:
            check()
        except (AssertionError, ValueError):
            return name
    return None


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    src = open(SRC).read()
    lib = _build(src, str(tmp_path), "control")
    assert _first_failing_pin(lib, monkeypatch) is None


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_fails_a_pin(mutant, tmp_path, monkeypatch):
    old, new = MUTANTS[mutant]
    src = open(SRC).read()
    assert src.count(old) == 1, f"{mutant}: the text to mutate must occur exactly once"
    lib = _build(src.replace(old, new), str(tmp_path), mutant)
    killed_by = _first_failing_pin(lib, monkeypatch)
    assert killed_by is not None, f"no pin catches the mutant {mutant}"
