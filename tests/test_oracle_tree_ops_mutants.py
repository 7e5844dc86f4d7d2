"""Pin strength for the oracle of the steps around verify: plant plausible mistakes in a
temporary copy of oracle/tree_ops.py and check that the pins in test_oracle_tree_ops.py
catch every one. The committed oracle is never changed.
"""
import importlib.util
import os

import pytest

from tests import test_oracle_tree_ops as P

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "tree_ops.py")

MUTANTS = {
    "rope_sin_sign_second_half": ("y[..., half:] = (x2 * c) + (x1 * s)", "y[..., half:] = (x2 * c) - (x1 * s)"),
    "rope_frequency_exponent": ("w = np.power(float(base), -2.0 * j / d)", "w = np.power(float(base), -1.0 * j / d)"),
    "rope_interleaved_pairs": ("x1, x2 = x[..., :half], x[..., half:]", "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    "rope_cos_sin_swapped": ("c = np.cos(a).astype(np.float32)", "c = np.sin(a).astype(np.float32)"),
    "positions_root_depth_one": ("depth[b, i] = 0 if p < 0 else depth[b, p] + 1",
                                 "depth[b, i] = 1 if p < 0 else depth[b, p] + 1"),
    "accept_child_own_target": ("int(tok[b, c]) == int(target[b, cur])", "int(tok[b, c]) == int(target[b, c])"),
    "accept_bonus_from_root": ("res.append((path, int(target[b, cur])))", "res.append((path, int(target[b, 0])))"),
    "accept_highest_index": ("                    nxt = c\n                    break\n", "                    nxt = c\n"),
    "compact_prefix_short": ("newp[b] = p0 + len(path)", "newp[b] = p0 + len(path) - 1"),
    "compact_source_unshifted": ("src_c = [np.array(c_kv[b, p0 + t]) for t in path]",
                                 "src_c = [np.array(c_kv[b, t]) for t in path]"),
    "build_tie_rank_before_parent": ("heapq.heappush(heap, (-float(sc), d, par, r, sc))",
                                     "heapq.heappush(heap, (-float(sc), d, r * 1000 + par, r, sc))"),
    "build_score_without_parent": ("sc = np.float32(score[b, par] + cand_lp[b, d - 1, k])",
                                   "sc = np.float32(cand_lp[b, d - 1, k])"),
    "build_depth_tie_ignored": ("heapq.heappush(heap, (-float(sc), d, par, r, sc))",
                                "heapq.heappush(heap, (-float(sc), 0, par, r, sc))"),
    "build_children_same_depth": ("push(n, d + 1, r2)", "push(n, d, r2)"),
    "vc_same_head_weights": ("v[..., h, :] = o64[..., h, :] @ w64[h]", "v[..., h, :] = o64[..., h, :] @ w64[0]"),
    "vc_latent_range_short": ("v[..., h, :] = o64[..., h, :] @ w64[h]",
                              "v[..., h, :] = o64[..., h, :448] @ w64[h, :448]"),
    "vc_other_head_latent": ("v[..., h, :] = o64[..., h, :] @ w64[h]",
                             "v[..., h, :] = o64[..., (h + 1) % H, :] @ w64[h]"),
    "vc_widen_shift": ("astype(np.uint32) << np.uint32(16)).view(np.float32)",
                       "astype(np.uint32) << np.uint32(15)).view(np.float32)"),
    "vc_weight_rows_reversed": ("v[..., h, :] = o64[..., h, :] @ w64[h]",
                                "v[..., h, :] = o64[..., h, :] @ w64[h, ::-1]"),
}

PINS = [
    (P.test_rope_matches_complex_exponential_form, dict(d=8, base=10000.0)),
    (P.test_rope_known_value_single_pair, {}),
    (P.test_rope_position_zero_is_identity, {}),
    (P.test_rope_preserves_pair_norms, {}),
    (P.test_rope_scores_depend_only_on_position_difference, {}),
    (P.test_rope_composes_additively, {}),
    (P.test_positions_on_chain_star_and_random_trees, {}),
    (P.test_accept_equals_brute_force_on_random_trees, dict(seed=7)),
    (P.test_accept_all_match_chain_and_no_match_root, {}),
    (P.test_accept_prefers_lowest_index_among_equal_sibling_tokens, {}),
    (P.test_compact_chain_path_is_identity, {}),
    (P.test_compact_moves_named_rows_and_nothing_else, {}),
    (P.test_build_equals_brute_force_selection_order, dict(seed=2, D=4, K=3, quant=True)),
    (P.test_build_invariants_and_single_candidate_chain, {}),
    (P.test_vc_one_hot_weights_select_latent_dims_exactly, {}),
    (P.test_vc_unit_latent_returns_weight_row, {}),
    (P.test_vc_triangular_closed_forms, {}),
    (P.test_vc_bf16_weights_widen_exactly, {}),
]


def _mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    f = tmp_path / f"tree_ops_{name}.py"
    f.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"tree_ops_mutant_{name}", str(f))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, monkeypatch, name):
    mod = _mutant(tmp_path, name, *MUTANTS[name])
    monkeypatch.setattr(P, "ot", mod)
    caught = []
    for pin, kw in PINS:
        try:
            pin(**kw)
        except Exception:                  # a failed check, or the mutant breaking outright
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
