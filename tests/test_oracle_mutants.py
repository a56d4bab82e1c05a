"""The oracle's pins catch plausible mistakes.

Each case copies the oracle to a temporary directory, plants one mistake in
its C source (a dropped term, a wrong sign or index, a swapped operand, a
wrong rounding), builds it, and runs the pin tests against the mutant: at
least one pin must fail. Nothing here touches the real oracle or the GPU."""
import importlib.util
import os
import shutil
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE = os.path.join(os.path.dirname(HERE), "oracle")

MUTANTS = {
    "bias dropped": ("int b = c + ORC_BIAS;", "int b = c;"),
    "v sign flipped": ("float v = u[j * ORC_CHUNK + i] - mu;", "float v = mu - u[j * ORC_CHUNK + i];"),
    "scale rounded down": ("s_h = orc_f16_from_double((double)s, 1);", "s_h = orc_f16_from_double((double)s, 0);"),
    "no sign-aware rule": ("return -(q > 1 ? q : 1);", "return -q;"),
    "nibbles swapped": ("((unsigned)a0 & 15u) | (((unsigned)a1 & 15u) << 4)",
                        "((unsigned)a1 & 15u) | (((unsigned)a0 & 15u) << 4)"),
    "threshold offset": ("(k - 0.5) / ORC_QMAX", "(k - 0.4) / ORC_QMAX"),
    "range not min-relative": ("rng = mx - mn;", "rng = mx;"),
    "mean over 32 slots": ("float mean = slot[0] / (float)nc;", "float mean = slot[0] / 32.0f;"),
    "anchor not at residual centre": ("    int c = 16 * A;\n    if (full)", "    int c = 16 * A + 7;\n    if (full)"),
    "residual bias dropped in decode": ("c = 16 * A + r - ORC_BIAS;", "c = 16 * A + r;"),
    "chunk sum left to right": ("for (int h = ORC_CHUNK / 2; h >= 1; h /= 2)\n                    for (int i = 0; i < h; ++i)\n"
                                "                        slot[i] = slot[i] + slot[i + h];",
                                "for (int i = 1; i < ORC_CHUNK; ++i)\n                    slot[0] = slot[0] + slot[i];"),
    "u by division": ("(bf16_to_f32(x[(size_t)t * ORC_D + d]) - mn) * inv_r;",
                      "(bf16_to_f32(x[(size_t)t * ORC_D + d]) - mn) / rng;"),
    "w by division": ("float w = v * inv_s;", "float w = sf > 0.0f ? v / sf : 0.0f;"),
    "mean times the reciprocal count": ("float mean = slot[0] / (float)nc;",
                                        "float mean = slot[0] * (1.0f / (float)nc);"),
    "GQA head mapping": ("const uint16_t *qh = q + ((size_t)b * Hq + (size_t)g * G + h) * ORC_D;",
                         "const uint16_t *qh = q + ((size_t)b * Hq + (size_t)h * H + g) * ORC_D;"),
}


def _mutant(tmp_path, name, old, new):
    d = tmp_path / "oracle_mut"
    shutil.copytree(ORACLE, d, ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    src = d / "lynx_oracle.c"
    text = src.read_text()
    assert text.count(old) >= 1, f"mutation site not found: {name}"
    src.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mut_{abs(hash(name))}", d / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


def _pins():
    """Cheapest first; a mutant is caught by the first one that fails."""
    import test_closed_forms as C
    import test_oracle_attention as A
    import test_oracle_encoder as E
    import test_oracle_map as M
    import test_oracle_contract_order as O
    import test_oracle_tables as T
    return [
        lambda o: T.test_thresholds_sit_at_half_levels(o),
        lambda o: T.test_tables_match_golden_fixture(o),
        lambda o: M.test_split_enumerates_all_codes(o),
        lambda o: M.test_sign_aware_mapping_keeps_small_negatives_negative(o),
        lambda o: C.test_structural_constants(o),
        lambda o: E.test_nibble_layout_even_channel_low(o),
        lambda o: E.test_residual_centre_gives_anchor_decode(o),
        lambda o: E.test_metadata_against_fp64_statistics(o),
        lambda o: E.test_ragged_chunk_metadata_against_fp64_statistics(o),
        lambda o: E.test_reconstruction_within_half_a_log_step(o),
        lambda o: E.test_brute_force_code_selection(o, 11),
        lambda o: O.test_u_is_a_product_with_the_reciprocal(o),
        lambda o: O.test_chunk_sum_is_the_stride_halving_tree(o),
        lambda o: O.test_w_is_a_product_with_the_reciprocal(o),
        lambda o: O.test_mean_is_a_division_by_the_valid_count(o),
        lambda o: A.test_gqa_groups_are_contiguous(o),
        lambda o: A.test_matches_numpy_softmax_through_permuted_pages(o, True),
        lambda o: M.test_map_is_round_half_up_in_log_domain(o),
    ]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    sys.path.insert(0, HERE)
    old, new = MUTANTS[name]
    mod = _mutant(tmp_path, name, old, new)
    for pin in _pins():
        try:
            pin(mod)
        except (AssertionError, ValueError):
            return
    raise AssertionError(f"no pin caught the mutant '{name}'")
