"""Planted mistakes in the CPU oracle must each fail a pin.

Every mutant below edits one expression of one oracle function -- a dropped
scale, a wrong sign, base or index, an off-by-one in a mask, swapped operands
-- recompiles that function against the oracle module's own globals and
patches it in for one test.  The named pin (from ``test_oracle_pins``) must
then fail.  A mutant whose text no longer occurs in the oracle is an error,
so the list cannot silently go stale as the oracle changes.

This runs on the CPU only and touches nothing outside the oracle module.
"""
import __future__
import inspect
import textwrap

import numpy as np
import pytest

from oracle import oracle as orc

import test_oracle_packed_pins as packed_pins
import test_oracle_pins as pins


def _plant(monkeypatch, fn_name: str, old: str, new: str) -> None:
    """Replace the one occurrence of ``old`` by ``new`` in ``orc.<fn_name>``."""
    src = textwrap.dedent(inspect.getsource(getattr(orc, fn_name)))
    assert src.count(old) == 1, f"mutant text not found exactly once in {fn_name}: {old!r}"
    code = compile(src.replace(old, new), f"<mutant of {fn_name}>", "exec",
                   flags=__future__.annotations.compiler_flag, dont_inherit=True)
    scope: dict = {}
    exec(code, orc.__dict__, scope)                     # globals: the live oracle module
    monkeypatch.setattr(orc, fn_name, scope[fn_name])
    if fn_name == "_e4m3_value":                         # the table is built from it at import
        monkeypatch.setattr(orc, "E4M3_TABLE",
                            np.array([scope[fn_name](c) for c in range(256)], dtype=np.float64))
    if fn_name == "_e2m1_value":
        monkeypatch.setattr(orc, "E2M1_TABLE",
                            np.array([scope[fn_name](c) for c in range(16)], dtype=np.float64))


def _split2():
    pins.test_split_combine_matches_unsplit(2)


def _dense_bf16():
    pins.test_dense_case_equals_torch_sdpa("bf16")


# (id, oracle function, original text, planted text, pin that must fail)
MUTANTS = [
    # element formats
    ("bf16_wrong_shift", "bf16_to_f64", "<< np.uint32(16)", "<< np.uint32(15)",
     pins.test_bf16_decode_matches_torch_for_every_code),
    ("e4m3_bias_8", "_e4m3_value", "2.0 ** (e - 7)", "2.0 ** (e - 8)",
     pins.test_e4m3_decode_matches_torch_for_every_code),
    ("e4m3_subnormal_implicit_one", "_e4m3_value", "(m / 8.0) * 2.0 ** -6", "(1.0 + m / 8.0) * 2.0 ** -6",
     pins.test_e4m3_decode_matches_torch_for_every_code),
    ("e4m3_no_nan", "_e4m3_value", "if e == 0xF and m == 0x7:", "if False:",
     pins.test_e4m3_decode_matches_torch_for_every_code),
    # packed KV rows
    ("e2m1_bias_0", "_e2m1_value", "2.0 ** (e - 1)", "2.0 ** e",
     packed_pins.test_e2m1_decode_matches_the_specification_for_every_code),
    ("e2m1_subnormal_implicit_one", "_e2m1_value", "return sign * m * 0.5", "return sign * (1.0 + m) * 0.5",
     packed_pins.test_e2m1_decode_matches_the_specification_for_every_code),
    ("ue8m0_bias_128", "ue8m0_to_f64", "- 127.0", "- 128.0", packed_pins.test_ue8m0_is_a_power_of_two_exponent),
    ("packed_fp8_blocks_reversed", "decode_packed_fp8_rows", "np.repeat(scale, 64, axis=1)",
     "np.repeat(scale[:, ::-1], 64, axis=1)", packed_pins.test_packed_fp8_row_closed_form),
    ("packed_fp8_rope_shifted", "decode_packed_fp8_rows", "rows[:, 456:584]", "rows[:, 454:582]",
     packed_pins.test_packed_fp8_row_closed_form),
    ("nvfp4_high_nibble_first", "decode_nvfp4_rows", "codes[:, 0::2] = packed & 0x0F",
     "codes[:, 0::2] = packed >> 4", packed_pins.test_nvfp4_row_closed_form),
    ("nvfp4_blocks_reversed", "decode_nvfp4_rows", "np.repeat(block, 16, axis=1)",
     "np.repeat(block[:, ::-1], 16, axis=1)", packed_pins.test_nvfp4_row_closed_form),
    ("nvfp4_row_scale_dropped", "decode_nvfp4_rows", "* np.repeat(block, 16, axis=1) * row_scale",
     "* np.repeat(block, 16, axis=1)", packed_pins.test_nvfp4_row_closed_form),
    ("nvfp4_rope_shifted", "decode_nvfp4_rows", "rows[:, 252:380]", "rows[:, 256:384]",
     packed_pins.test_nvfp4_row_closed_form),
    ("packed_query_as_e4m3", "decode", 'if dtype in ("bf16", "packed_fp8", "nvfp4"):',
     'if dtype in ("bf16",):', packed_pins.test_single_slot_through_an_nvfp4_row),
    ("packed_rows_decoded_as_bf16", "decode_rows", 'if dtype == "packed_fp8":', 'if dtype == "packed":',
     packed_pins.test_single_slot_through_a_packed_fp8_row),
    # token metadata
    ("dense_tokens_strided", "token_request", "return t // q_len, t % q_len, q_len",
     "return t % batch, t // batch, q_len", pins.test_varlen_right_aligned_positions),
    ("varlen_bounds_shifted", "token_request", "if cum[b] <= t < cum[b + 1]:",
     "if cum[b] < t <= cum[b + 1]:", pins.test_varlen_right_aligned_positions),
    ("left_aligned_position", "token_position", "int(seq_lens[b]) - q_len + i",
     "int(seq_lens[b]) - 1 - i", pins.test_varlen_right_aligned_positions),
    # slot selection
    ("swa_window_off_by_one", "valid_slots", "- q_len + i + 1))", "- q_len + i))",
     pins.test_swa_window_reading),
    ("swa_window_ignored", "valid_slots", "if idx == -1 or j >= w_swa:", "if idx == -1:",
     pins.test_swa_window_reading),
    ("swa_topk_lens_ignored", "valid_slots", "w_swa = min(max(int(swa_topk_lens[t]), 0), SWA_COLS)",
     "w_swa = SWA_COLS", pins.test_swa_topk_lens_equals_minus_one_mask),
    ("topk_off_by_one", "valid_slots", "for j in range(n_lim):", "for j in range(n_lim - 1):",
     pins.test_topk_lens_mask_equals_minus_one_mask),
    ("topk_not_clamped_low", "valid_slots", "min(max(int(topk_lens[t]), 0), width)",
     "min(abs(int(topk_lens[t])), width)", pins.test_topk_lens_mask_equals_minus_one_mask),
    ("minus_one_in_compressed_kept", "valid_slots",
     "idx = int(indices[t, j])\n            if idx == -1:\n                continue\n            pool, rows = \"comp\"",
     "idx = int(indices[t, j])\n            pool, rows = \"comp\"", pins.test_fully_masked_token_is_zero_with_minus_inf_lse),
    ("invalid_index_masked_silently", "valid_slots", 'if invalid_index == "raise":', "if False:",
     pins.test_invalid_index_raises_or_masks),
    ("page_and_offset_swapped", "valid_slots",
     "comp_block_tables[t, c // comp_page_size]) * comp_page_size + c % comp_page_size",
     "comp_block_tables[t, c % comp_page_size]) * comp_page_size + c // comp_page_size",
     pins.test_page_table_slots_golden),
    ("hca_count_without_window", "valid_slots", "int(hca_seq_lens[b]) - SWA_COLS", "int(hca_seq_lens[b])",
     pins.test_page_table_slots_golden),
    ("block_table_row_by_request", "valid_slots", "comp_block_tables[t, c // comp_page_size]",
     "comp_block_tables[b, c // comp_page_size]", pins.test_page_table_is_indexed_by_token),
    # gathering
    ("duplicates_collapsed", "_gather", "rows = [pool_bits[p][r] for (_, p, r) in slots]",
     "rows = [pool_bits[p][r] for (p, r) in dict.fromkeys((p, r) for (_, p, r) in slots)]",
     pins.test_duplicate_index_counts_twice),
    ("swa_rows_read_from_comp_pool", "_gather", "pool_bits[p][r]", "pool_bits['comp'][r % len(pool_bits['comp'])]",
     _dense_bf16),
    # attention for one token
    ("bmm1_dropped", "attend", "logits = bmm1 * (q_t @ kv.T)", "logits = (q_t @ kv.T)",
     pins.test_two_slot_worked_example),
    ("logits_in_base_2", "attend", "e = np.exp(logits - m[:, None])", "e = np.exp2(logits - m[:, None])",
     _dense_bf16),
    ("bmm2_dropped", "attend", "o = bmm2 * (e @ kv)", "o = (e @ kv)",
     pins.test_single_valid_slot_returns_row_times_bmm2),
    ("sink_scaled_by_bmm1", "attend", "np.exp(np.asarray(sinks, dtype=np.float64) - m)",
     "np.exp(bmm1 * np.asarray(sinks, dtype=np.float64) - m)", pins.test_single_valid_slot_returns_row_times_bmm2),
    ("sink_sign_flipped", "attend", "np.exp(np.asarray(sinks, dtype=np.float64) - m)",
     "np.exp(-np.asarray(sinks, dtype=np.float64) - m)", pins.test_equal_logit_sink_closed_form),
    ("sink_in_lse", "attend", "np.log(denom if lse_with_sink else z)", "np.log(denom)",
     pins.test_single_valid_slot_returns_row_times_bmm2),
    ("lse_natural_log", "attend", "* LOG2E", "* 1.0", pins.test_two_slot_worked_example),
    ("lse_missing_max", "attend", "lse2 = (m + np.log(", "lse2 = (np.log(", pins.test_two_slot_worked_example),
    ("max_not_subtracted", "attend", "e = np.exp(logits - m[:, None])", "e = np.exp(logits)",
     pins.test_dominant_logit_selects_its_row_without_overflow),
    ("sink_dropped_from_normaliser", "attend", "o = bmm2 * (e @ kv) / denom[:, None]",
     "o = bmm2 * (e @ kv) / z[:, None]", pins.test_sink_limits),
    ("bmm2_applied_twice", "attend", "o = bmm2 * (e @ kv)", "o = bmm2 * bmm2 * (e @ kv)",
     pins.test_output_is_linear_in_bmm2_and_lse_ignores_it),
    ("bmm1_squared", "attend", "logits = bmm1 * (q_t @ kv.T)", "logits = bmm1 * bmm1 * 8.0 * (q_t @ kv.T)",
     pins.test_power_of_two_query_scale_trades_with_bmm1),
    ("pv_rows_reversed", "attend", "(e @ kv)", "(e @ kv[::-1])", pins.test_two_slot_worked_example),
    ("softmax_over_heads", "attend", "m = logits.max(axis=1)", "m = logits.max(axis=1).max()",
     pins.test_zero_query_gives_mean_and_log2_n),
    # split partials and their combine
    ("combine_weights_natural_exp", "combine_partials", "np.exp2(lse_s - mx_safe[None, :])",
     "np.exp(lse_s - mx_safe[None, :])", pins.test_combine_of_two_partials_closed_form),
    ("combine_lse_natural_log", "combine_partials", "mx_safe[ok] + np.log2(wsum[ok])",
     "mx_safe[ok] + np.log(wsum[ok])", pins.test_combine_of_two_partials_closed_form),
    ("combine_sink_not_rescaled", "combine_partials", "sink2 = np.asarray(sinks, dtype=np.float64) * LOG2E",
     "sink2 = np.asarray(sinks, dtype=np.float64)", _split2),
    ("combine_bmm2_dropped", "combine_partials", "return bmm2 * out, lse", "return out, lse", _split2),
    ("combine_empty_split_not_skipped", "combine_partials",
     "np.where(np.isfinite(lse_s), np.exp2(lse_s - mx_safe[None, :]), 0.0)",
     "np.exp2(np.where(np.isfinite(lse_s), lse_s, 0.0) - mx_safe[None, :])",
     pins.test_combine_of_two_partials_closed_form),
    ("split_ranges_overlap", "sparse_mla_decode", "min(n_lim, (s + 1) * per)", "min(n_lim, (s + 2) * per)",
     _split2),
]


@pytest.mark.parametrize("mid, fn, old, new, pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_planted_mistake(monkeypatch, mid, fn, old, new, pin):
    pin()                                                # the pin holds on the oracle as written
    _plant(monkeypatch, fn, old, new)
    with pytest.raises((AssertionError, IndexError, ValueError, pytest.fail.Exception)):
        pin()


def test_mutant_ids_are_unique():
    ids = [m[0] for m in MUTANTS]
    assert len(ids) == len(set(ids))


def test_pins_catch_a_dropped_sink(monkeypatch):
    """Plant a mistake in the oracle (sink left out) and check a pin fails."""
    orig = orc.attend
    monkeypatch.setattr(orc, "attend", lambda q, kv, b1, b2, s, lse_with_sink=False: orig(q, kv, b1, b2, None))
    with pytest.raises(AssertionError):
        pins.test_equal_logit_sink_closed_form()


def test_pins_catch_a_transposed_contraction(monkeypatch):
    """Plant a mistake (PV uses the logits' softmax over heads, not slots)."""
    def bad(q_t, kv, bmm1, bmm2, sinks, lse_with_sink=False):
        o, lse = orig(q_t, kv, bmm1, bmm2, sinks, lse_with_sink)
        if kv.shape[0] == 0 or q_t.shape[0] < 2:
            return o, lse
        logits = bmm1 * (q_t @ kv.T)
        e = np.exp(logits - logits.max(axis=0, keepdims=True))
        return bmm2 * (e / e.sum(axis=0, keepdims=True)) @ kv, lse
    orig = orc.attend
    monkeypatch.setattr(orc, "attend", bad)
    with pytest.raises(AssertionError):
        pins.test_dense_case_equals_torch_sdpa("bf16")
