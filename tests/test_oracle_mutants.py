"""Plant plausible mistakes in copies of the oracle source; each must fail a pin.

This is how the pins are shown to pin something: a dropped term, a wrong sign or
index, a transposed operand or a reversed tie rule anywhere in the oracle has to
be caught.  The mutants are compiled from text substitutions into a temporary
directory; the oracle itself is never modified."""
import os

import pytest

import oracle
import oracle_pins

# (name, original text, replacement) or (name, [(original, replacement), ...]).
# Every original must occur exactly once.
MUTANTS = [
    ("topk_tie_toward_higher_id",
     "return (a->id > b->id) - (a->id < b->id);", "return (a->id < b->id) - (a->id > b->id);"),
    ("topk_margin_from_top1",
     "(double)c[K - 1].val - (double)c[K].val", "(double)c[0].val - (double)c[K].val"),
    ("logits_reversed_operand",
     "acc += bf16_value(h[p * D + d]) * bf16_value(W_lm[v * D + d]);",
     "acc += bf16_value(h[p * D + d]) * bf16_value(W_lm[v * D + (D - 1 - d)]);"),
    ("logits_dropped_last_term",
     "            for (int64_t d = 0; d < D; ++d)\n                acc += bf16_value(h[p * D + d]) * bf16_value(W[v * D + d]);",
     "            for (int64_t d = 0; d + 1 < D; ++d)\n                acc += bf16_value(h[p * D + d]) * bf16_value(W[v * D + d]);"),
    ("G_wrong_row",
     "bf16_value(W_H[(int64_t)i * D + d])", "bf16_value(W_H[(int64_t)(r - 1 - i) * D + d])"),
    ("walk_no_feedback", "            a = best_id;", "            a = anchors[q];"),
    ("walk_tie_toward_higher_id", "(s == best && b < best_id)", "(s == best && b > best_id)"),
    ("pair_drops_context_gate", "* (double)Grow[i] *", "*"),
    ("pair_sign_flip", "        s += bf16_value(A[", "        s -= bf16_value(A["),
    ("walk_gate_from_previous_row",
     "float s = pair_score(vals[row * K + j], a, b, G + row * r, A, Bc, r);",
     "float s = pair_score(vals[row * K + j], a, b, G + (row - 1) * r, A, Bc, r);"),
    ("pair_wrong_predecessor", "        int32_t a = pred[p];", "        int32_t a = ids[p * K];"),
    ("walk_margin_unflagged_ties", "                } else if (s > second) {", "                } else if (s > second && s < best) {"),
    ("conv_crosses_block",
     "                if (t - j < 0) continue;\n                double k = (double)base[((int64_t)0",
     "                if (p - j < 0) continue;\n                double k = (double)base[((int64_t)0"),
    ("conv_group_strided",
     "d[((int64_t)0 * taps + j) * G + c / g];", "d[((int64_t)0 * taps + j) * G + c % G];"),
    ("conv_proj_io_j_swapped",
     "d[((int64_t)0 * taps + j) * G + c / g];", "d[((int64_t)j * 2 + 0) * G + c / g];"),
    ("conv_tap_reads_current_row",
     "acc += k * act_value(x, x_is_f32, (p - j) * C + c);", "acc += k * act_value(x, x_is_f32, p * C + c);"),
    ("conv_finish_uses_input_base",
     "double k = (double)base[((int64_t)1 * taps + j) * C + c] +",
     "double k = (double)base[((int64_t)0 * taps + j) * C + c] +"),
    ("conv_finish_ignores_dynamic",
     "(double)dyn_out[(p * taps + j) * G + c / g];", "0.0 * (double)dyn_out[(p * taps + j) * G + c / g];"),
    ("conv_dyn_out_from_input_side",
     "(float)d[((int64_t)1 * taps + j) * G + gi];", "(float)d[((int64_t)0 * taps + j) * G + gi];"),
    ("bf16_double_rounding", "    if (lo == 0x8000u) {", "    if (0) {"),
    ("conv_no_validation", "P % Bsz == 0;", "1;"),
    ("lattice_predecessor_from_same_row",
     "a = ids[(row - 1) * K + i];", "a = ids[row * K + i];"),
    ("lattice_first_slot_reads_anchor_row",
     "a = anchors[q];\n                } else {", "a = ids[(row - 1) * K];\n                } else {"),
    ("lattice_gate_from_previous_row",
     "ids[row * K + j], G + row * r", "ids[row * K + j], G + (row - 1) * r"),
    ("lattice_walk_no_feedback", "            i = pick;", "            i = 0;"),
    ("lattice_walk_tie_toward_higher_id",
     "(s == best && cand[j] < cand[pick])", "(s == best && cand[j] > cand[pick])"),
    ("lattice_walk_margin_unflagged_ties",
     "} else if (second < s) {", "} else if (second < s && s < best) {"),
    ("sampling_ignores_temperature",
     "w[j] = exp(((double)Lrow[j] - mx) / temperature);", "w[j] = exp(((double)Lrow[j] - mx));"),
    ("sampling_reflected_uniform",
     "if (below + w[j] > u * total) {", "if (below + w[j] > (1.0 - u) * total) {"),
    ("sampling_margin_wrong_end",
     "if (pick > 0) mg = u - lo / total;", "if (pick > 0) mg = u - hi / total;"),
    ("softcap_no_outer_cap",
     "return cap > 0.0 ? cap * tanh(x / cap) : x;", "return cap > 0.0 ? tanh(x / cap) : x;"),
    ("softcap_multiplier_after_cap",
     "return cap > 0.0 ? cap * tanh(x / cap) : x;", "return cap > 0.0 ? mul * cap * tanh(u / cap) : x;"),
    ("softcap_multiplier_dropped", "const double x = mul * u;", "const double x = u;"),
    ("softcap_scaled_not_divided",
     "return cap > 0.0 ? cap * tanh(x / cap) : x;", "return cap > 0.0 ? cap * tanh(x * cap) : x;"),
    ("softcap_after_selection", [
        ("c[v].val = (float)logit_map(acc, mul, cap);", "c[v].val = (float)acc;"),
        ("vals[p * K + j] = c[j].val;", "vals[p * K + j] = (float)logit_map(c[j].val, mul, cap);")]),
    ("softcap_accepts_negative_multiplier", "if (!(mul > 0.0) ||", "if (!(mul != 0.0) ||"),
    ("finish_prepare_drops_residual", "    if (residual) {\n", "    if (0) {\n"),
    ("finish_prepare_next_reads_z",
     "return df2o_conv_prepare(h, is_f32,", "return df2o_conv_prepare(z, is_f32,"),
    ("finish_prepare_next_uses_same_base",
     "W_proj, base_next, y_next, dyn_next);", "W_proj, base, y_next, dyn_next);"),
    ("ce_sign_flip",
     "loss[p] = (float)(log(sum) + m - (double)scores[p * K + js]);",
     "loss[p] = (float)(log(sum) + m + (double)scores[p * K + js]);"),
    ("ce_max_shift_not_restored",
     "loss[p] = (float)(log(sum) + m - (double)scores[p * K + js]);",
     "loss[p] = (float)(log(sum) - (double)scores[p * K + js]);"),
    ("ce_label_is_the_best_column",
     "                if (ids[p * K + j] == y) {", "                if (scores[p * K + j] >= scores[p * K] && ids[p * K + j] != -7) {"),
    ("ce_uncovered_rows_count_zero", "            loss[p] = NAN;\n            continue;", "            loss[p] = 0.0f;\n            continue;"),
    ("ce_sum_skips_last", "        for (int32_t j = 0; j < K; ++j) sum += exp(", "        for (int32_t j = 0; j + 1 < K; ++j) sum += exp("),
    ("ce_no_status_for_large_target", "        if (y >= V) bad |= 1;\n", "        if (0) bad |= 1;\n"),
    ("ce_label_off_by_one",
     "loss[p] = (float)(log(sum) + m - (double)scores[p * K + js]);",
     "loss[p] = (float)(log(sum) + m - (double)scores[p * K + (js + 1) % K]);"),
    # transposed operands and off-by-one rows in the selector
    ("pair_codebooks_swapped",
     "bf16_value(A[(int64_t)a * r + i]) * (double)Grow[i] * bf16_value(Bc[(int64_t)b * r + i])",
     "bf16_value(A[(int64_t)b * r + i]) * (double)Grow[i] * bf16_value(Bc[(int64_t)a * r + i])"),
    ("pair_drops_unary", "    double s = (double)u;\n", "    double s = 0.0 * (double)u;\n"),
    ("walk_reads_previous_row",
     "            const int64_t row = (int64_t)q * Bsz + t;\n            float best = -INFINITY, second = -INFINITY;",
     "            const int64_t row = (int64_t)q * Bsz + t - 1;\n            float best = -INFINITY, second = -INFINITY;"),
    ("walk_margin_reversed",
     "margin[q * T + (t - 1)] = (K > 1) ? (double)best - (double)second : INFINITY;",
     "margin[q * T + (t - 1)] = (K > 1) ? (double)second - (double)best : INFINITY;"),
    ("lattice_slot0_rows_zero",
     "for (int32_t j = 0; j < K; ++j) Lt[(int64_t)i * K + j] = NAN;",
     "for (int32_t j = 0; j < K; ++j) Lt[(int64_t)i * K + j] = 0.0f;"),
    ("lattice_walk_row_stride", " + (int64_t)i * K;", " + (int64_t)i;"),
    ("lattice_walk_path_is_column", "path[q * T + (t - 1)] = cand[pick];", "path[q * T + (t - 1)] = pick;"),
    ("sampling_margin_counts_end_one", "if (pick < K - 1 && hi / total - u < mg)", "if (hi / total - u < mg)"),
    ("sampling_margin_counts_end_zero", "if (pick > 0) mg = u - lo / total;", "mg = u - lo / total;"),
    # the head: margin sign, a cap of 0, G from one row, fp32 accumulation
    ("topk_margin_sign", "(double)c[K - 1].val - (double)c[K].val", "(double)c[K].val - (double)c[K - 1].val"),
    ("softcap_zero_cap_applies",
     "return cap > 0.0 ? cap * tanh(x / cap) : x;", "return cap >= 0.0 ? cap * tanh(x / cap) : x;"),
    ("G_reads_first_row",
     "acc += bf16_value(h[p * D + d]) * bf16_value(W_H[(int64_t)i * D + d]);",
     "acc += bf16_value(h[d]) * bf16_value(W_H[(int64_t)i * D + d]);"),
    ("logits_fp32_accumulate",
     "            double acc = 0.0;\n            for (int64_t d = 0; d < D; ++d)\n"
     "                acc += bf16_value(h[p * D + d]) * bf16_value(W[v * D + d]);",
     "            float acc = 0.0f;\n            for (int64_t d = 0; d < D; ++d)\n"
     "                acc += (float)(bf16_value(h[p * D + d]) * bf16_value(W[v * D + d]));"),
    # the conv: reversed taps, one tap's correction, corrections of the wrong row
    ("conv_base_taps_reversed",
     "double k = (double)base[((int64_t)0 * taps + j) * C + c] +",
     "double k = (double)base[((int64_t)0 * taps + (taps - 1 - j)) * C + c] +"),
    ("conv_dyn_out_tap0_only",
     "dyn_out[(p * taps + j) * G + gi] = (float)d[((int64_t)1 * taps + j) * G + gi];",
     "dyn_out[(p * taps + j) * G + gi] = (float)d[((int64_t)1 * taps + 0) * G + gi];"),
    ("conv_finish_dyn_from_source_row",
     "(double)dyn_out[(p * taps + j) * G + c / g];", "(double)dyn_out[((p - j) * taps + j) * G + c / g];"),
    ("conv_projection_reads_block_start",
     "acc += bf16_value(W_proj[n * C + c]) * act_value(x, x_is_f32, p * C + c);",
     "acc += bf16_value(W_proj[n * C + c]) * act_value(x, x_is_f32, (p - p % Bsz) * C + c);"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


def _sites(m):
    """A mutant's (original, replacement) pairs: one site, or a list of them."""
    return m[1] if len(m) == 2 else [(m[1], m[2])]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, mutant):
    name = mutant[0]
    mutated = source
    for orig, repl in _sites(mutant):
        assert source.count(orig) == 1, f"mutation site for {name} not unique/found"
        mutated = mutated.replace(orig, repl)
    src = tmp_path / f"{name}.c"
    src.write_text(mutated)
    lib = oracle.build(str(src), str(tmp_path / f"lib{name}.so"), force=True)
    o = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
