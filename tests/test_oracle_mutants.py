"""The oracle's pins must catch plausible mistakes.

Each case below plants one slip in a copy of oracle.c (on the CPU only),
compiles it to a temporary library, points the oracle binding at it and runs
a battery of the pin tests.  A mutant survives if every pin still passes;
the test fails if any mutant survives.
"""
import ctypes
import os
import subprocess

import pytest

import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.c")

# (name, original text, planted text[, how many occurrences]); default: all
MUTANTS = [
    ("bias_dropped", "+ bias_at(D, b, h, q, k);", ";"),
    ("ds_sign", "double dS = P * (dP - Dq);", "double dS = P * (dP + Dq);"),
    ("gqa_head_map", "int g = h / G;", "int g = h % D->Hkv;"),
    ("window_left_off_by_one", "k < q + off - D->window_left) return 0;", "k <= q + off - D->window_left) return 0;"),
    ("window_right_range", "z = c + D->window_right;", "z = c + D->window_right - 1;"),
    ("causal_excludes_diagonal", "if (D->causal && k > q + off) return 0;", "if (D->causal && k >= q + off) return 0;"),
    ("varlen_keys_not_cut", "if (q >= lq || k >= lk) return 0;", "if (q >= lq) return 0;"),
    ("bottom_right_offset_sign", "*off = D->bottom_right ? nk - nq : 0;", "*off = D->bottom_right ? nq - nk : 0;"),
    ("sink_left_out_of_denominator", "double l = with_sink ? exp(sk - m) : 0.0;", "double l = 0.0;"),
    ("sink_left_out_of_max", "if (sk > m) m = sk;", "if (sk > m && any) m = sk;"),
    ("sink_gradient_sign", "ds_part[b * D->Hq + h] -= exp(", "ds_part[b * D->Hq + h] += exp("),
    ("dropout_one_word_per_call", "return out[k & 3];", "return out[0];"),
    ("dropout_counter_without_head", "(uint32_t)q, (uint32_t)h, (uint32_t)b};", "(uint32_t)q, 0u, (uint32_t)b};"),
    ("dropout_keeps_the_dropped", "drop_draw(D, b, h, q, k) < D->drop_threshold) return 0;",
     "drop_draw(D, b, h, q, k) >= D->drop_threshold) return 0;"),
    ("dropout_not_applied", "if (D->drop_threshold && drop_draw(D, b, h, q, k) < D->drop_threshold) return 0;", ";"),
    # slips inside the generator keep it a bijection with good statistics; only its
    # published known answers catch them
    ("philox_round_constant", "(uint64_t)0xD2511F53u * c[0]", "(uint64_t)0xD2511F55u * c[0]"),
    ("philox_weyl_increment", "k1 += 0xBB67AE85u;", "k1 += 0xBB67AE87u;"),
    ("philox_hi_lo_swapped", "const uint32_t n1 = (uint32_t)pb;", "const uint32_t n1 = (uint32_t)(pb >> 32) ^ 1u;"),
    ("select_nan_order_of_visit", "if (best < 0 || ranks_above(sc[j], sc[best])) best = j;",
     "if (best < 0 || sc[j] > sc[best]) best = j;"),
    ("philox_nine_rounds", "for (int r = 0; r < 10; ++r) {", "for (int r = 0; r < 9; ++r) {"),
    ("dk_transposed_operand", "dkr[c] = dkr[c] + D->scale * dS * qrow[c];",
     "dkr[c] = dkr[c] + D->scale * dS * kr[c];", 1),
    ("dq_scale_dropped", "dqrow[c] = dqrow[c] + D->scale * dS * kr[c];", "dqrow[c] = dqrow[c] + dS * kr[c];"),
    ("dv_missing_p", "dvr[c] = dvr[c] + P * dorow[c];", "dvr[c] = dvr[c] + dorow[c];"),
    ("denominator_unshifted", "l = l + exp(z[k] - m);", "l = l + exp(z[k]);"),
    ("carry_correction_dropped", "nr[c] = nr[c] * corr;", "nr[c] = nr[c];"),
    ("carry_denominator_uncorrected", "den[r] = den[r] * corr + rs;", "den[r] = den[r] + rs;"),
    # the visiting order of the ring changes rounding only, so the planted
    # slip is a ring that revisits its own KV block instead of rotating
    ("ring_does_not_rotate", "int j = ((i - idx) % n + n) % n;", "int j = i;"),
    ("select_ties_upper", "    return a > b;\n}", "    return a >= b;\n}"),
    ("local_window_wide", "(k >= q - (D->local_window - 1))", "(k >= q - D->local_window)"),
    ("union_drops_selected", "if (sel[t] >= 0 && k / D->sel_block == sel[t]) in_sel = 1;",
     "if (sel[t] >= 0 && k / D->sel_block == sel[t] + 1) in_sel = 1;"),
]
# (a selection that also considers its own block needs several edits: below)


def battery(ora):
    yield lambda: [pins.test_closed_form_fixture(ora, c) for c in pins._golden()["cases"]]
    yield lambda: pins.test_closed_form_gradient_fixture(ora)
    for mask in pins.MASKS:
        yield lambda mask=mask: pins.test_fwd_matches_brute_force(ora, mask, (4, 2), "full")
    yield lambda: pins.test_gqa_equals_repeated_heads(ora)
    yield lambda: pins.test_gradients_match_finite_differences(
        ora, dict(causal=True, window=(3, 0), bias=True))
    yield lambda: pins.test_window_00_is_identity_and_gradients(ora)
    yield lambda: pins.test_key_gradients_sum_to_zero(ora)
    yield lambda: pins.test_blockwise_carry_equals_one_shot(ora, 2, dict(causal=True, window=(-1, -1)))
    yield lambda: pins.test_blockwise_carry_equals_one_shot(ora, 4, dict(causal=False, window=(-1, -1)))
    yield lambda: pins.test_select_matches_full_sort(ora, "f64")
    yield lambda: pins.test_select_planted_ranking(ora)
    yield lambda: pins.test_select_ties_keep_lower_block(ora)
    yield lambda: pins.test_select_fewer_candidates_than_top_n(ora)
    yield lambda: pins.test_select_nan_scores_rank_last(ora)
    yield lambda: pins.test_block_selected_attention_matches_brute_force(ora)
    for case in pins.VARLEN_CASES:
        yield lambda case=case: pins.test_varlen_matches_rebuilt_problems(ora, case, dict(causal=True, window=(3, 0)))
    yield lambda: pins.test_varlen_padding_is_inert(ora)
    yield lambda: pins.test_sink_equals_extra_key(ora, True, "learnable")
    yield lambda: pins.test_sink_rows_without_keys_and_padding(ora)
    yield lambda: pins.test_sink_gradients_match_finite_differences(ora)
    yield lambda: pins.test_philox_known_answers(ora)
    yield lambda: pins.test_dropout_draws_are_bernoulli(ora, 0.1)
    yield lambda: pins.test_dropout_is_the_fixed_mask(ora, True)


def _build_mutant(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    lib = tmp_path / f"lib{name}.so"
    src.write_text(text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-o", str(lib), str(src), "-lm"], check=True)
    return str(lib)


def _killed(ora, lib_path):
    saved = ora._lib
    ora._lib = ora._bind(ctypes.CDLL(lib_path))
    try:
        for check in battery(ora):
            try:
                check()
            except AssertionError:
                return True
        return False
    finally:
        ora._lib = saved


def test_unmutated_copy_passes_battery(ora, tmp_path):
    with open(SRC) as f:
        lib = _build_mutant(tmp_path, "clean", f.read())
    assert not _killed(ora, lib)


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(ora, tmp_path, mutant):
    name, old, new = mutant[:3]
    count = mutant[3] if len(mutant) > 3 else -1
    with open(SRC) as f:
        text = f.read()
    assert old in text, f"mutation site for {name} not found"
    lib = _build_mutant(tmp_path, name, text.replace(old, new, count))
    assert _killed(ora, lib), f"mutant {name} survived every pin"


def test_mutant_select_own_block_is_caught(ora, tmp_path):
    with open(SRC) as f:
        text = f.read()
    old1 = "for (int j = 0; j < i; ++j) sc[j] = dot("
    old2 = "int take = i < top_n ? i : top_n;"
    old3 = "for (int j = 0; j < i; ++j) pick[j] = 0;"
    assert old1 in text and old2 in text and old3 in text
    t = text.replace(old1, "for (int j = 0; j <= i && j < nblk; ++j) sc[j] = dot(")
    t = t.replace(old2, "int take = i + 1 < top_n ? i + 1 : top_n;")
    t = t.replace(old3, "for (int j = 0; j <= i; ++j) pick[j] = 0;")
    t = t.replace("for (int j = 0; j < i; ++j) {\n                            if (pick[j]) continue;",
                  "for (int j = 0; j <= i; ++j) {\n                            if (pick[j]) continue;")
    t = t.replace("for (int j = 0; j < i; ++j)\n                        if (pick[j]) dst[w++] = j;",
                  "for (int j = 0; j <= i; ++j)\n                        if (pick[j]) dst[w++] = j;")
    lib = _build_mutant(tmp_path, "own_block", t)
    assert _killed(ora, lib)
