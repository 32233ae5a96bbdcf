"""Planted mistakes in the oracle must fail one of its pins.

Each mutant is a copy of mlora_oracle.c with one plausible mistake (a dropped term, a wrong
sign, a transposed operand, a wrong index, a rounding slip). The copy is built in a temporary
directory and run through the pins of ``oracle_pins``; the test passes when some pin rejects
the mutant. The real oracle is never modified. Every mutant keeps all accesses in bounds.
"""
import os

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    "scale_dropped": ("double out = orc_decode(y_row[n], p->dtype) + sc * acc;",
                      "double out = orc_decode(y_row[n], p->dtype) + acc;"),
    "delta_sign": ("double out = orc_decode(y_row[n], p->dtype) + sc * acc;",
                   "double out = orc_decode(y_row[n], p->dtype) - sc * acc;"),
    "base_y_dropped": ("double out = orc_decode(y_row[n], p->dtype) + sc * acc;", "double out = sc * acc;"),
    "scale_of_slot0": ("double sc = (double)p->scale[s];", "double sc = (double)p->scale[0];"),
    "segment_bounds_shifted": ("if (off[t] <= i && i < off[t + 1]) return seg_slot[t];",
                               "if (off[t] < i && i <= off[t + 1]) return seg_slot[t];"),
    "expand_uses_r_max": ("int r = p->rank[s];\n  double sc", "int r = p->r_max;\n  double sc"),
    "layer_ignored": ("((size_t)s * (size_t)p->num_layers + (size_t)layer)", "((size_t)s * (size_t)p->num_layers + 0)"),
    "a_transposed": ("return orc_decode(p->a_t[row * (size_t)p->d_in + (size_t)k], p->dtype);",
                     "return orc_decode(p->a_t[(row - (size_t)j) * (size_t)p->d_in + (size_t)k * (size_t)p->r_max"
                     " + (size_t)j], p->dtype);"),
    "b_transposed": ("return orc_decode(p->b[row * (size_t)p->d_out + (size_t)n], p->dtype);",
                     "return orc_decode(p->b[(row - (size_t)j) * (size_t)p->d_out + (size_t)n * (size_t)p->r_max"
                     " + (size_t)j], p->dtype);"),
    "b_page_from_a_table": ("int32_t page = p->b_page_table[", "int32_t page = p->a_page_table["),
    "minus_one_uses_slot0": ("if (s == -1) return 0; /* no adapter: the row is not touched */", "if (s == -1) s = 0;"),
    "last_k_dropped": ("for (int k = 0; k < p->d_in; ++k)", "for (int k = 0; k < p->d_in - 1; ++k)"),
    "last_j_dropped": ("for (int j = 0; j < r; ++j) acc += v_row[j]", "for (int j = 0; j < r - 1; ++j) acc += v_row[j]"),
    "ties_away_from_zero": ("(rem == 0.5 && fmod(fl, 2.0) != 0.0)", "(rem == 0.5)"),
    "truncating_round": ("if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;", ""),
    "subnormal_decode_off_by_one": ("ldexp((double)m, 1 - f.bias - f.mant_bits)", "ldexp((double)m, -f.bias - f.mant_bits)"),
    "overflow_threshold_low": ("if (r >= ldexp(1.0, emax + 1))", "if (r > ldexp(1.0, emax))"),
    "bgmv_slot_of_next_row": ("int32_t s = off ? sgmv_row_slot(off, seg_slot, nseg, i) : row_slot[i];",
                              "int32_t s = off ? sgmv_row_slot(off, seg_slot, nseg, i) : row_slot[i + 1 < M ? i + 1 : i];"),
    "shrink_drops_top_rank_row": ("int r = p->rank[s];\n  for (int j = 0; j < r; ++j) {\n    double acc = 0.0;",
                                  "int r = p->rank[s] - 1;\n  for (int j = 0; j < r; ++j) {\n    double acc = 0.0;"),
    "page_of_vector_start_only": ("  return table_index(p, s, layer, j) * (size_t)pages_per_vector(p, d) + (size_t)(k / p->page_elems);",
                                  "  return table_index(p, s, layer, j) * (size_t)pages_per_vector(p, d) + (size_t)(k / p->page_elems) * 0;"),
    "page_entry_of_next_vector_piece": ("  return table_index(p, s, layer, j) * (size_t)pages_per_vector(p, d) + (size_t)(k / p->page_elems);",
                                        "  return table_index(p, s, layer, j) * (size_t)pages_per_vector(p, d) + (size_t)((k / p->page_elems + 1) % pages_per_vector(p, d));"),
    "x_element_shifted": ("acc += orc_decode(x_row[k], p->dtype) * elem_a(p, s, layer, k, j);",
                          "acc += orc_decode(x_row[k > 0 ? k - 1 : 0], p->dtype) * elem_a(p, s, layer, k, j);"),
}

# the operator pins run first: they are cheap and catch most mutants
ORDER = [P.pin_rank_closed_form, P.pin_slot_identification, P.pin_identical_is_dense_gemm, P.pin_merged_identity,
         P.pin_skip_rows_untouched, P.pin_status_contract, P.pin_sampled_rows, P.pin_sgmv_equals_bgmv_on_the_same_rows,
         P.pin_vectors_across_pages_equal_stacked, P.pin_round_ties,
         P.pin_round_trip_exhaustive, P.pin_decode_exhaustive, P.pin_round_matches_library]


def test_mutation_list_is_complete():
    assert set(ORDER) == set(P.ALL_PINS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) == 1, f"mutation target for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(before, after))
    lib = oracle.load(oracle.build(force=True, src=str(path), out=str(tmp_path / f"lib{name}.so")))
    for pin in ORDER:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            return
    pytest.fail(f"mutant {name} passed every pin")
