"""Pins for the CPU oracle: each checks it against something other than itself.

- visibility: exhaustive brute force (closure by boolean matrix products) on every
  tree with T <= 6, chain and star shapes, word padding, bad-parent detection;
- attention: torch float64 softmax (a library routine) on causal (chain tree),
  dense (all-visible) and arbitrary tree masks; explicit path sets on every tree
  with T <= 5; the closed form for a zero query (tests/golden); single-key
  exactness; weights sum to one with exact zeros elsewhere; prefix-permutation
  invariance; split-prefix LSE merge equals the unsplit result.
"""
import math

import numpy as np
import pytest

import workloads as wl
from tests import helpers as H

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- visibility --

@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6])
def test_visibility_exhaustive(oracle_mod, T):
    trees = list(H.all_parent_arrays(T))
    assert len(trees) == math.factorial(T)
    parents = np.stack(trees)
    got = oracle_mod.build_visibility(parents)
    want = np.stack([H.pack_bits(H.closure_visible(p)) for p in trees])
    assert got.dtype == np.uint32 and got.shape == (len(trees), T, 1)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("T", [1, 31, 32, 33, 64, 65, 128])
def test_visibility_chain_star_and_padding(oracle_mod, T):
    W = (T + 31) // 32
    chain = oracle_mod.build_visibility(wl.tree_chain(T)[None])[0]
    star = oracle_mod.build_visibility(wl.tree_star(T)[None])[0]
    for i in range(T):
        bits_chain = [(chain[i, t // 32] >> (t % 32)) & 1 for t in range(32 * W)]
        bits_star = [(star[i, t // 32] >> (t % 32)) & 1 for t in range(32 * W)]
        assert bits_chain == [1 if t <= i else 0 for t in range(32 * W)]      # lower triangular
        assert bits_star == [1 if (t == 0 or t == i) else 0 for t in range(32 * W)]


def test_visibility_rejects_bad_parent(oracle_mod):
    p = np.stack([wl.tree_chain(8), wl.tree_chain(8)])
    p[1, 5] = 5          # not < i
    with pytest.raises(oracle_mod.OracleError, match="flat index 13"):
        oracle_mod.build_visibility(p)
    p[1, 5] = 4
    p[0, 3] = -2         # < -1
    with pytest.raises(oracle_mod.OracleError, match="flat index 3"):
        oracle_mod.build_visibility(p)


# ------------------------------------------------------------------ attention --

def _small(T=5, H=2, prefix=3, dtype="f32", tree="uniform", seed=7, B=2, **kw):
    return wl.make_case("t", B=B, T=T, H=H, prefix=prefix, dtype=dtype, tree=tree, seed=seed, **kw)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chain_tree_equals_causal_attention(oracle_mod, dtype):
    case = _small(T=9, H=3, prefix=11, dtype=dtype, tree="chain")
    out, lse = oracle_mod.verify_attn_rows(case, np.arange(case.rows), f64=True)
    # causal: tree query i sees every cache row j < prefix + i + 1
    mask = np.zeros((case.B, case.T, case.L), dtype=bool)
    for b in range(case.B):
        for i in range(case.T):
            mask[b, i, :case.prefix_len[b] + i + 1] = True
    ro, rl = H.torch_reference(case, mask)
    np.testing.assert_allclose(out.reshape(ro.shape), ro, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(rl.shape), rl, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_visible_equals_dense_attention(oracle_mod, dtype):
    case = _small(T=7, H=2, prefix=(5, 9), dtype=dtype)
    W = case.W
    vis = np.zeros((case.B, case.T, W), dtype=np.uint32)
    vis[..., 0] = (1 << case.T) - 1
    out, lse = oracle_mod.verify_attn_rows(case, np.arange(case.rows), vis=vis, f64=True)
    mask = np.zeros((case.B, case.T, case.L), dtype=bool)
    for b in range(case.B):
        mask[b, :, :case.prefix_len[b] + case.T] = True
    ro, rl = H.torch_reference(case, mask)
    np.testing.assert_allclose(out.reshape(ro.shape), ro, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(rl.shape), rl, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("tree", ["uniform", "geometric", "depth16", "window8"])
def test_tree_masks_match_library_softmax(oracle_mod, tree):
    case = _small(T=40, H=2, prefix=(3, 17), dtype="bf16", tree=tree, seed=11)
    out, lse = oracle_mod.verify_attn_rows(case, np.arange(case.rows), f64=True)
    ro, rl = H.torch_reference(case, H.tree_key_mask(case))
    np.testing.assert_allclose(out.reshape(ro.shape), ro, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(rl.shape), rl, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5])
def test_every_tiny_tree_matches_explicit_path_sets(oracle_mod, T):
    # Brute force: every tree with T nodes, two prefix lengths, visible set from the
    # closure (not the oracle's walk), library softmax over exactly those rows.
    for k, parent in enumerate(H.all_parent_arrays(T)):
        case = wl.make_case("p", B=2, T=T, H=2, prefix=(0, 2), dtype="f32", tree=parent, seed=100 + k)
        out, lse = oracle_mod.verify_attn_rows(case, np.arange(case.rows), f64=True)
        ro, rl = H.torch_reference(case, H.tree_key_mask(case))
        np.testing.assert_allclose(out.reshape(ro.shape), ro, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse.reshape(rl.shape), rl, rtol=1e-12, atol=1e-13)


def test_golden_zero_query_closed_form(oracle_mod):
    for g in H.read_golden_cases("q_zero_uniform.txt"):
        T = len(g["parent"])
        case = wl.make_case(g["name"], B=1, T=T, H=3, prefix=g["prefix"], dtype="f32",
                            tree=g["parent"], seed=5)
        case.q_nope[:] = 0
        case.q_pe[:] = 0
        out, lse = oracle_mod.verify_attn(case)
        ck = H.widen(case.c_kv[0], "f32")
        for i in range(T):
            np.testing.assert_allclose(lse[0, i], math.log(g["count"][i]), rtol=1e-6)
            if i in g["paths"]:
                rows = list(range(g["prefix"])) + [g["prefix"] + t for t in g["paths"][i]]
                assert len(rows) == g["count"][i]
                np.testing.assert_allclose(out[0, i], np.broadcast_to(ck[rows].mean(0), out[0, i].shape),
                                           rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_visible_key_is_exact(oracle_mod, dtype):
    # prefix 0: the root (query 0) sees only itself -> p = 1, o = c_kv[row] exactly.
    case = _small(T=6, H=4, prefix=0, dtype=dtype, seed=3)
    out, lse = oracle_mod.verify_attn(case)
    ck = H.widen(case.c_kv, dtype)
    kp = H.widen(case.k_pe, dtype)
    qn = H.widen(case.q_nope, dtype)
    qp = H.widen(case.q_pe, dtype)
    for b in range(case.B):
        for h in range(case.H):
            np.testing.assert_array_equal(out[b, 0, h].astype(np.float64), ck[b, 0])
            s = case.scale * (np.dot(qn[b, 0, h], ck[b, 0]) + np.dot(qp[b, 0, h], kp[b, 0]))
            np.testing.assert_allclose(lse[b, 0, h], s, rtol=1e-6, atol=1e-6)
    # a caller-supplied mask that shows one tree key t to query i
    vis = np.zeros((case.B, case.T, 1), dtype=np.uint32)
    for i in range(case.T):
        vis[:, i, 0] = 1 << ((3 * i + 1) % case.T)
    out, _ = oracle_mod.verify_attn(case, vis=vis)
    for i in range(case.T):
        np.testing.assert_array_equal(out[:, i, 0].astype(np.float64), ck[:, (3 * i + 1) % case.T])


def test_weights_sum_to_one_and_vanish_off_the_visible_set(oracle_mod):
    case = _small(T=20, H=2, prefix=(4, 13), dtype="bf16", tree="geometric", seed=9)
    mask = H.tree_key_mask(case)
    for row in range(0, case.rows, 3):
        p = oracle_mod.attn_weights(case, row)
        b, i = row // (case.T * case.H), (row // case.H) % case.T
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.all(p[~mask[b, i]] == 0.0)
        assert np.all(p[mask[b, i]] > 0.0)


def test_empty_visible_set_gives_zero_and_minus_inf(oracle_mod):
    case = _small(T=4, H=2, prefix=0, seed=4)
    vis = np.zeros((case.B, case.T, 1), dtype=np.uint32)
    vis[0, 1, 0] = 0b0010
    out, lse = oracle_mod.verify_attn(case, vis=vis)
    assert np.isneginf(lse[1]).all() and (out[1] == 0).all()
    assert np.isneginf(lse[0, 0]).all() and np.isfinite(lse[0, 1]).all()


def test_padding_rows_are_never_read(oracle_mod):
    case = _small(T=8, H=2, prefix=(3, 30), dtype="bf16", seed=12)   # sequence 0 padded with NaN
    out, lse = oracle_mod.verify_attn(case)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_prefix_permutation_invariance(oracle_mod):
    case = _small(T=6, H=2, prefix=25, dtype="f32", seed=21)
    out, lse = oracle_mod.verify_attn_rows(case, np.arange(case.rows), f64=True)
    perm = np.random.default_rng(0).permutation(25)
    case.c_kv[:, :25] = case.c_kv[:, perm]
    case.k_pe[:, :25] = case.k_pe[:, perm]
    out2, lse2 = oracle_mod.verify_attn_rows(case, np.arange(case.rows), f64=True)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-14)


def test_split_prefix_merge_equals_unsplit(oracle_mod):
    # Attention over (first half of prefix + tree) merged by log-sum-exp with
    # attention over (second half of prefix) must equal the full result.
    full = _small(T=6, H=2, prefix=40, dtype="f32", seed=31, B=1)
    out, lse = oracle_mod.verify_attn_rows(full, np.arange(full.rows), f64=True)
    P, T = 40, 6
    a = wl.make_case("a", B=1, T=T, H=2, prefix=20, dtype="f32", tree=full.parent, seed=31)
    a.q_nope[:], a.q_pe[:] = full.q_nope, full.q_pe
    a.c_kv[0, :20], a.k_pe[0, :20] = full.c_kv[0, :20], full.k_pe[0, :20]
    a.c_kv[0, 20:20 + T], a.k_pe[0, 20:20 + T] = full.c_kv[0, P:P + T], full.k_pe[0, P:P + T]
    bcase = wl.make_case("b", B=1, T=T, H=2, prefix=20, dtype="f32", tree=full.parent, seed=31)
    bcase.q_nope[:], bcase.q_pe[:] = full.q_nope, full.q_pe
    bcase.c_kv[0, :20], bcase.k_pe[0, :20] = full.c_kv[0, 20:40], full.k_pe[0, 20:40]
    oa, la = oracle_mod.verify_attn_rows(a, np.arange(a.rows), f64=True)
    ob, lb = oracle_mod.verify_attn_rows(bcase, np.arange(bcase.rows),
                                         vis=np.zeros((1, T, 1), np.uint32), f64=True)
    om, lm = oracle_mod.merge_states(oa, la, ob, lb)
    np.testing.assert_allclose(om, out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lm, lse, rtol=1e-12, atol=1e-13)


def test_merge_states_edge_cases(oracle_mod):
    o_a = np.ones((3, 4))
    o_b = 2 * np.ones((3, 4))
    la = np.array([-np.inf, 0.0, -np.inf])
    lb = np.array([-np.inf, -np.inf, 1.5])
    o, l = oracle_mod.merge_states(o_a, la, o_b, lb)
    assert np.isneginf(l[0]) and (o[0] == 0).all()
    assert l[1] == 0.0 and (o[1] == 1).all()
    assert l[2] == 1.5 and (o[2] == 2).all()
    # equal weights average the states: lse grows by ln 2
    o, l = oracle_mod.merge_states(o_a[:1], np.array([0.3]), o_b[:1], np.array([0.3]))
    np.testing.assert_allclose(o, 1.5)
    np.testing.assert_allclose(l, 0.3 + math.log(2.0))


def test_bf16_widening_is_exact(oracle_mod):
    case = _small(T=1, H=1, prefix=0, dtype="bf16", seed=2, B=1)
    pats = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000], dtype=np.uint16)   # 1, -2, min subnormal, max, -0
    case.c_kv[0, 0, :5] = pats
    out, _ = oracle_mod.verify_attn(case)
    want = H.widen(pats, "bf16")
    np.testing.assert_array_equal(out[0, 0, 0, :5].astype(np.float64), want)


def test_generator_is_deterministic_and_shaped():
    a = wl.make_config("tiny")
    b = wl.make_config("tiny")
    np.testing.assert_array_equal(a.q_nope, b.q_nope)
    assert a.L == 46 and a.kv_len.tolist() == [46, 46]
    assert a.parent[:, 0].tolist() == [-1, -1]
    for p in a.parent:
        assert all(0 <= p[i] < i for i in range(1, a.T))
    x = wl.normal(3, "x", 200000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    # bf16 rounding: exact values stay, ties go to even
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], dtype=np.float64)
    np.testing.assert_array_equal(wl.f64_to_bf16_bits(v), np.array([0x3F80, 0x3F80, 0x3F82, 0xC020], np.uint16))
