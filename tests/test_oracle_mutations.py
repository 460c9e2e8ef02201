"""Plant plausible mistakes in a temporary copy of the oracle and check that the
pins in test_oracle_pins.py catch every one of them.  CPU only.

Each mutant is the oracle's C source with one textual edit, compiled with gcc
into a temporary directory and swapped in for the duration of one check.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sfa_oracle.c")

# (name, original text, planted text, pins expected to catch it)
MUTANTS = [
    ("dropped_scale", "double s = p->scale * dot;", "double s = dot;",
     [pins.test_single_entry_gives_that_row_and_its_scaled_score]),
    ("log2_lse", "*lse_out = m + log(l);", "*lse_out = m + log2(l);",
     [pins.test_zero_query_gives_mean_of_selected_rows_and_ln_k]),
    ("v_from_rope_side", "out_row[c] += w * bf16_to_double(vrow[c]);",
     "out_row[c] += w * bf16_to_double(vrow[c + 64]);",
     [pins.test_zero_query_gives_mean_of_selected_rows_and_ln_k]),
    ("score_skips_rope", "for (int d = 0; d < p->D; ++d) dot +=",
     "for (int d = 0; d < p->DV; ++d) dot +=",
     [pins.test_rope_columns_enter_the_score_but_not_the_output]),
    ("causal_off_by_one", "return (long)p->seq_lens[b] - (long)(p->Q - 1 - i);",
     "return (long)p->seq_lens[b] - (long)(p->Q - i);",
     [pins.test_mtp_query_tokens_see_their_own_causal_range]),
    ("interleave_group_of_block", "if (p->interleave > 0 && n > 1 && r >= 0) return (pos / p->interleave) % n == r;",
     "if (p->interleave > 0 && n > 1 && r >= 0) return (pos / p->block_size) % n == r;",
     [pins.test_interleaved_shard_partials_closed_form_with_zero_query]),
    ("bt_row_per_sequence_always", "int b = p->bt_per_token ? t : t / p->Q;   /* block-table row */",
     "int b = t / p->Q;   /* block-table row */",
     [pins.test_block_table_per_token_reads_each_tokens_own_row]),
    ("slot_ignores_table", "return phys * p->block_size + pos % p->block_size;",
     "return (long)row * p->max_blocks_per_seq * p->block_size + pos;",
     [pins.test_physical_block_placement_does_not_matter]),
    ("slot_offset_swapped", "return phys * p->block_size + pos % p->block_size;",
     "return phys * p->block_size + (pos / p->block_size) % p->block_size;",
     [pins.test_one_hot_rows_recover_the_exact_multiset_read]),
    ("shard_floor", "long c = S > 0 ? (S + n - 1) / n : 0;", "long c = S > 0 ? S / n : 0;",
     [pins.test_shard_partials_closed_form_with_zero_query]),
    ("merge_weight_sign", "double w = exp(lse_part[(size_t)r * rows + x] - L);",
     "double w = exp(L - lse_part[(size_t)r * rows + x]);",
     [pins.test_merge_identity_order_and_empty_partials]),
    ("no_dedup_semantics", "long pos = idx[j];\n    if (!in_unit(p, pos, lo, hi, n_sh, r)) continue;",
     "long pos = idx[j];\n    if (!in_unit(p, pos, lo, hi, n_sh, r)) continue;\n    if (j > 0 && idx[j - 1] == pos) continue;",
     [pins.test_duplicate_entries_count_once_per_list_entry]),
    ("kv_write_next_slot", "for (int d = 0; d < D; ++d) kv[(size_t)s * D + d] = rows[(size_t)t * D + d];",
     "for (int d = 0; d < D; ++d) kv[(size_t)(s + 1 < num_slots ? s + 1 : s) * D + d] = rows[(size_t)t * D + d];",
     [pins.test_kv_write_places_rows_skips_padding_and_leaves_the_rest,
      pins.test_decode_after_write_reads_the_new_token_row]),
    ("kv_write_writes_padding",
     "    const long s = slot_mapping[t];\n    if (s < 0) continue;\n    for (int d = 0; d < D; ++d)",
     "    const long s = slot_mapping[t] < 0 ? 0 : slot_mapping[t];\n    for (int d = 0; d < D; ++d)",
     [pins.test_kv_write_places_rows_skips_padding_and_leaves_the_rest]),
    ("topk_ties_higher_position_first", "return a->pos < b->pos ? -1 : (a->pos > b->pos ? 1 : 0);",
     "return a->pos > b->pos ? -1 : (a->pos < b->pos ? 1 : 0);",
     [pins.test_topk_ties_take_lower_positions_first]),
    ("topk_ignores_causal_range", "if (causal < L) L = causal;", "(void)causal;",
     [pins.test_topk_causal_range_and_short_rows]),
    ("topk_negatives_like_positives", "  return ma > mb ? -1 : 1;\n}", "  return ma < mb ? -1 : 1;\n}",
     [pins.test_topk_signed_zero_infinities_and_nan_follow_total_order, pins.test_topk_distinct_scores_match_numpy_sort]),
    ("topk_signed_zeros_equal", "if (neg_a != neg_b) return neg_a ? -1 : 1;",
     "if (neg_a != neg_b && ((a | b) & 0x7FFFFFFFu)) return neg_a ? -1 : 1;",
     [pins.test_topk_signed_zero_infinities_and_nan_follow_total_order]),
    ("topk_output_in_score_order", "qsort(sel, (size_t)n, sizeof(int32_t), pos_ascending);", "(void)pos_ascending;",
     [pins.test_topk_distinct_scores_match_numpy_sort]),
    ("padding_minus_one_only", "if (!in_unit(p, pos, lo, hi, n_sh, r)) continue;\n    long slot = slot_of(p, b, pos);\n    if (slot < 0) return -1;",
     "if (pos == -1) continue;\n    long slot = slot_of(p, b, pos);\n    if (slot < 0) return -1;",
     [pins.test_empty_selection_gives_zero_and_minus_inf]),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)  # every occurrence: both passes over the list
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"lib{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(c_path),
                    "-o", str(so_path), "-lm"], check=True)
    return oracle._bind(str(so_path))


@pytest.mark.parametrize("name,old,new,catchers", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name, old, new, catchers):
    lib = _build_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(oracle, "_lib", lib)
    for catch in catchers:
        caught = False
        try:
            catch()
        except (AssertionError, RuntimeError):
            caught = True
        assert caught, f"pin {catch.__name__} did not catch mutant {name}"
