"""Pin strength: plant plausible mistakes in a copy of the oracle and check that the
pins in test_oracle.py catch every one. The mutation is made in a temporary copy of
the C source on the CPU; the committed oracle is never changed.
"""
import importlib.util
import os
import shutil

import pytest

from tests import test_oracle as P

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_DIR = os.path.join(os.path.dirname(HERE), "oracle")

MUTANTS = {
    "rope_term_dropped": ("dot += ld(a->q_pe, a->dtype, qrow * DR + d) * ld(a->k_pe, a->dtype, krow * DR + d);",
                          "dot += 0.0;"),
    "self_not_visible": ("visible[P + j] = 1;", "if (j != i) visible[P + j] = 1;"),
    "prefix_off_by_one": ("for (long long j = 0; j < P; ++j) visible[j] = 1;",
                          "for (long long j = 1; j < P; ++j) visible[j] = 1;"),
    "root_not_walked": ("while (j >= 0) {                                       /* self + ancestors */",
                        "while (j > 0) {"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "weights_unnormalised": ("double p = exp(s[j] - m) / l;", "double p = exp(s[j] - m);"),
    "head_query_transposed": ("size_t qrow = ((size_t)b * a->T + i) * a->H + h;",
                              "size_t qrow = ((size_t)b * a->H + h) * a->T + i;"),
    "bit_order_reversed": ("w[j / 32] |= (uint32_t)1u << (j % 32);", "w[j / 32] |= (uint32_t)1u << (31 - j % 32);"),
    "scale_dropped": ("s[j] = a->scale * dot;", "s[j] = dot;"),
    "merge_weights_swapped": ("(wa * o_a[(size_t)r * D + d] + wb * o_b", "(wb * o_a[(size_t)r * D + d] + wa * o_b"),
    "bits_input_off_by_one": ("if ((w[t / 32] >> (t % 32)) & 1u) visible[P + t] = 1;",
                              "if ((w[t / 32] >> (t % 32)) & 1u) visible[P + t + (t + 1 < a->T)] = 1;"),
}

PINS = [
    (P.test_visibility_exhaustive, dict(T=5)),
    (P.test_visibility_chain_star_and_padding, dict(T=33)),
    (P.test_chain_tree_equals_causal_attention, dict(dtype="f32")),
    (P.test_all_visible_equals_dense_attention, dict(dtype="bf16")),
    (P.test_tree_masks_match_library_softmax, dict(tree="geometric")),
    (P.test_every_tiny_tree_matches_explicit_path_sets, dict(T=3)),
    (P.test_golden_zero_query_closed_form, {}),
    (P.test_single_visible_key_is_exact, dict(dtype="f32")),
    (P.test_weights_sum_to_one_and_vanish_off_the_visible_set, {}),
    (P.test_split_prefix_merge_equals_unsplit, {}),
    (P.test_merge_states_edge_cases, {}),
]


def _mutant_module(tmp_path, name, old, new):
    src = open(os.path.join(ORACLE_DIR, "kdt_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    d = tmp_path / name
    d.mkdir()
    (d / "kdt_oracle.c").write_text(src.replace(old, new))
    shutil.copy(os.path.join(ORACLE_DIR, "__init__.py"), d / "__init__.py")
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}", str(d / "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    mod = _mutant_module(tmp_path, name, old, new)
    caught = []
    for fn, kw in PINS:
        try:
            fn(mod, **kw)
        except Exception as e:       # an assertion or an oracle error both count as caught
            caught.append((fn.__name__, type(e).__name__))
    assert caught, f"no pin caught mutant {name}"
