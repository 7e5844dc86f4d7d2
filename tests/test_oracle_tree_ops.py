"""Pins for the oracle of the steps around tree-verify attention (CPU only).

Each check ties the oracle to something other than its own formula: the complex form of
the rotation, invariants RoPE is built to have, brute force over tree paths, and row by
row comparisons with the rows a path names.
"""
import numpy as np
import pytest

import workloads as wl
from oracle import tree_ops as ot


def _vecs(seed, n, d):
    return wl.normal(seed, "rope_x", n * d).reshape(n, d)


# ------------------------------------------------------------------ RoPE pins --
@pytest.mark.parametrize("d,base", [(2, 10000.0), (8, 10000.0), (64, 10000.0), (64, 50000.0)])
def test_rope_matches_complex_exponential_form(d, base):
    # NeoX pairs element j with j + d/2: as a complex number z_j = x_j + i x_{j+d/2}, the
    # rotation multiplies z_j by exp(i p w_j), w_j = 1 / base^(2j/d). The oracle rounds
    # cos, sin, each product and each sum to float32: a few float32 ulps of the result's
    # scale apart from the exact value.
    x = _vecs(1, 40, d).astype(np.float32)
    pos = np.arange(40) * 37 + 3
    y = ot.rope_neox(x, pos, base).astype(np.float64)
    inv_freq = 1.0 / (base ** (np.arange(0, d, 2, dtype=np.float64) / d))
    z = (x[:, : d // 2] + 1j * x[:, d // 2:]).astype(np.complex128) * np.exp(1j * pos[:, None] * inv_freq[None, :])
    scale = np.abs(x).max()
    np.testing.assert_allclose(y[:, : d // 2], z.real, rtol=0, atol=4e-7 * scale)
    np.testing.assert_allclose(y[:, d // 2:], z.imag, rtol=0, atol=4e-7 * scale)


def test_rope_known_value_single_pair():
    # width 2: the only frequency is 1, so position 1 turns (1, 0) by one radian
    y = ot.rope_neox(np.array([[1.0, 0.0]]), np.array([1]), 10000.0)
    assert y.dtype == np.float32
    assert y[0].tolist() == [np.float32(0.5403023058681398), np.float32(0.8414709848078965)]


def test_rope_position_zero_is_identity():
    x = _vecs(2, 16, 64).astype(np.float32)
    assert np.array_equal(ot.rope_neox(x, np.zeros(16, dtype=np.int64), 10000.0), x)


def test_rope_preserves_pair_norms():
    x = _vecs(3, 32, 64).astype(np.float32)
    y = ot.rope_neox(x, np.arange(32) * 1000 + 17, 10000.0).astype(np.float64)
    x = x.astype(np.float64)
    nx = x[:, :32] ** 2 + x[:, 32:] ** 2
    ny = y[:, :32] ** 2 + y[:, 32:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=2e-6, atol=1e-7)


def test_rope_scores_depend_only_on_position_difference():
    q = _vecs(4, 8, 64).astype(np.float32)
    k = _vecs(5, 8, 64).astype(np.float32)
    m = np.array([0, 5, 100, 8192, 9000, 1, 77, 4096])
    n = np.array([3, 5, 90, 8000, 9000, 0, 70, 4100])
    dot = lambda a, b: np.sum(a.astype(np.float64) * b.astype(np.float64), axis=1)
    for shift in (1, 1000, 20000):
        a = dot(ot.rope_neox(q, m, 10000.0), ot.rope_neox(k, n, 10000.0))
        b = dot(ot.rope_neox(q, m + shift, 10000.0), ot.rope_neox(k, n + shift, 10000.0))
        np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-5)


def test_rope_composes_additively():
    x = _vecs(6, 12, 64).astype(np.float32)
    p = np.arange(12) * 311
    q = np.arange(12) * 97 + 5
    np.testing.assert_allclose(ot.rope_neox(ot.rope_neox(x, p, 10000.0), q, 10000.0),
                               ot.rope_neox(x, p + q, 10000.0), rtol=1e-5, atol=1e-5)


# --------------------------------------------------------------- positions --
def test_positions_on_chain_star_and_random_trees():
    assert ot.tree_positions(wl.tree_chain(5)[None], np.array([7])).tolist() == [[7, 8, 9, 10, 11]]
    assert ot.tree_positions(wl.tree_star(5)[None], np.array([7])).tolist() == [[7, 8, 8, 8, 8]]
    par = wl.tree_uniform(11, "pos", 40)
    pos = ot.tree_positions(par[None], np.array([100]))[0]
    for i in range(40):
        d, j = 0, i
        while par[j] >= 0:
            j = int(par[j])
            d += 1
        assert pos[i] == 100 + d


# ------------------------------------------------------------ accept pins --
def _distinct_sibling_tokens(par, seed):
    """Draft tokens in a 6-token alphabet with distinct tokens among siblings."""
    T = par.shape[0]
    tok = np.zeros(T, dtype=np.int64)
    perm = (wl.raw_u64(seed, "tok", T) % 6).astype(np.int64)
    used = {}
    for c in range(1, T):
        s = used.setdefault(int(par[c]), set())
        t = int(perm[c])
        while t in s:
            t = (t + 1) % 1000
        s.add(t)
        tok[c] = t
    return tok


def _brute_accept(par, tok, tgt):
    """Deepest node whose every root-path edge matches, by enumerating all nodes."""
    T = par.shape[0]
    best = 0
    best_depth = 0
    for i in range(T):
        ok, d, j = True, 0, i
        while par[j] >= 0:
            p = int(par[j])
            if tok[j] != tgt[p]:
                ok = False
                break
            j = p
            d += 1
        if ok and d > best_depth:
            best, best_depth = i, d
    path = [best]
    while par[path[-1]] >= 0:
        path.append(int(par[path[-1]]))
    return path[::-1], int(tgt[best])


@pytest.mark.parametrize("seed", range(12))
def test_accept_equals_brute_force_on_random_trees(seed):
    T = 3 + seed * 5
    par = (wl.tree_uniform(seed, "acc", T) if seed % 2 else wl.tree_geometric(seed, "acc", T))
    tok = _distinct_sibling_tokens(par, seed)
    tgt = (wl.raw_u64(seed, "tgt", T) % 4).astype(np.int64)    # small alphabet: matches happen
    (path, bonus), = ot.tree_accept(par[None], tok[None], tgt[None])
    assert (path, bonus) == _brute_accept(par, tok, tgt)


def test_accept_all_match_chain_and_no_match_root():
    T = 9
    par = wl.tree_chain(T)
    tgt = np.arange(T) + 100
    tok = np.concatenate([[0], tgt[:-1]])                        # node i drafts target[i-1]
    (path, bonus), = ot.tree_accept(par[None], tok[None], tgt[None])
    assert path == list(range(T)) and bonus == tgt[-1]
    tok2 = tok + 1
    (path, bonus), = ot.tree_accept(par[None], tok2[None], tgt[None])
    assert path == [0] and bonus == tgt[0]


# ----------------------------------------------------------- compaction pins --
def test_compact_chain_path_is_identity():
    c = wl.normal(1, "c", 2 * 20 * 8).reshape(2, 20, 8)
    k = wl.normal(2, "k", 2 * 20 * 4).reshape(2, 20, 4)
    pre = np.array([5, 9])
    c2, k2, newp = ot.kv_compact(c, k, pre, [[0, 1, 2], [0, 1, 2, 3, 4]])
    assert np.array_equal(c2, c) and np.array_equal(k2, k) and newp.tolist() == [8, 14]


def test_compact_moves_named_rows_and_nothing_else():
    B, L, T = 3, 40, 10
    c = wl.normal(3, "c", B * L * 8).reshape(B, L, 8)
    k = wl.normal(4, "k", B * L * 4).reshape(B, L, 4)
    pre = np.array([0, 7, 25])
    paths = [[0, 2, 5, 9], [0], [0, 1, 3]]
    c2, k2, newp = ot.kv_compact(c, k, pre, paths)
    assert newp.tolist() == [4, 8, 28]
    for b in range(B):
        n = len(paths[b])
        for r in range(L):
            if pre[b] <= r < pre[b] + n:
                src = pre[b] + paths[b][r - pre[b]]
                assert np.array_equal(c2[b, r], c[b, src]) and np.array_equal(k2[b, r], k[b, src])
            else:
                assert np.array_equal(c2[b, r], c[b, r]) and np.array_equal(k2[b, r], k[b, r])


def test_accept_prefers_lowest_index_among_equal_sibling_tokens():
    # the definition's tie rule: several children drafting the target's token -> lowest index
    par = np.array([-1, 0, 0, 0, 2, 3])
    tok = np.array([0, 5, 7, 7, 9, 9])
    tgt = np.array([7, 0, 9, 9, 1, 1])
    (path, bonus), = ot.tree_accept(par[None], tok[None], tgt[None])
    assert path == [0, 2, 4] and bonus == 1


# ------------------------------------------------------------- builder pins --
def _cands(seed, B, D, K, quant):
    """Distinct tokens per depth; log-probabilities <= 0, quantised to force score ties."""
    lp = -np.abs(wl.normal(seed, "lp", B * D * K)).reshape(B, D, K)
    if quant:
        lp = -np.round(-lp * 2.0) / 2.0
    tok = (np.arange(B * D * K).reshape(B, D, K) * 7 + 3).astype(np.int32)
    return tok, lp.astype(np.float32)


def _brute_build(tok, lp, N):
    """Every node of the full candidate tree (rank paths up to depth D), float32 path
    scores, sorted by the selection order with parents compared recursively; first N."""
    import functools
    D, K = lp.shape
    order = [sorted(range(K), key=lambda k: (-float(lp[d, k]), k)) for d in range(D)]
    score = {(): np.float32(0.0)}
    nodes = []
    frontier = [()]
    for d in range(1, D + 1):
        nxt = []
        for path in frontier:
            for r in range(K):
                p2 = path + (r,)
                score[p2] = np.float32(score[path] + lp[d - 1, order[d - 1][r]])
                nxt.append(p2)
        nodes += nxt
        frontier = nxt

    def cmp(a, b):
        if a == b:
            return 0
        if score[a] != score[b]:
            return -1 if score[a] > score[b] else 1
        if len(a) != len(b):
            return -1 if len(a) < len(b) else 1
        c = cmp(a[:-1], b[:-1]) if a[:-1] != b[:-1] else 0
        if c:
            return c
        return -1 if a[-1] < b[-1] else 1

    chosen = sorted(nodes, key=functools.cmp_to_key(cmp))[:N]
    index = {(): 0}
    for n, path in enumerate(chosen, start=1):
        index[path] = n
    par = [-1] + [index[p[:-1]] for p in chosen]
    tk = [-1] + [int(tok[len(p) - 1, order[len(p) - 1][p[-1]]]) for p in chosen]
    dep = [0] + [len(p) for p in chosen]
    sc = [np.float32(0.0)] + [score[p] for p in chosen]
    return par, tk, dep, sc


@pytest.mark.parametrize("seed,D,K,quant", [(0, 1, 3, False), (1, 3, 2, True), (2, 4, 3, True), (3, 3, 4, False),
                                            (4, 5, 2, True), (5, 2, 5, True)])
def test_build_equals_brute_force_selection_order(seed, D, K, quant):
    tok, lp = _cands(seed, 2, D, K, quant)
    total = sum(K ** d for d in range(1, D + 1))
    for N in sorted({1, total // 2, total}):
        par, tk, dep, sc = ot.tree_build(tok, lp, N)
        for b in range(2):
            ep, et, ed, es = _brute_build(tok[b], lp[b], N)
            assert par[b].tolist() == ep and tk[b].tolist() == et and dep[b].tolist() == ed
            assert np.array_equal(sc[b], np.array(es, dtype=np.float32))


def test_build_invariants_and_single_candidate_chain():
    tok, lp = _cands(9, 3, 6, 4, False)
    par, tk, dep, sc = ot.tree_build(tok, lp, 40, root_tok=np.array([5, 6, 7]))
    assert tk[:, 0].tolist() == [5, 6, 7]
    lp_of = {(b, int(tok[b, d, k])): lp[b, d, k] for b in range(3) for d in range(6) for k in range(4)}
    for b in range(3):
        for n in range(1, 41):
            p = par[b, n]
            assert 0 <= p < n and dep[b, n] == dep[b, p] + 1
            assert sc[b, n] == np.float32(sc[b, p] + lp_of[(b, int(tk[b, n]))])
        assert np.all(np.diff(sc[b]) <= 0)                     # log-probs <= 0: scores never rise
    tok1, lp1 = _cands(10, 1, 8, 1, False)
    par, tk, dep, sc = ot.tree_build(tok1, lp1, 8)
    assert par[0].tolist() == list(range(-1, 8)) and dep[0].tolist() == list(range(9))


# ----------------------------------------------------- w_vc up-projection pins --
def _bf16_bits(x):
    return wl.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def test_vc_one_hot_weights_select_latent_dims_exactly():
    # w_vc[h, d, n] = 1 iff d = sel[h, n]: v[r, h, n] = o[r, h, sel[h, n]], exactly, with a
    # different selection per head (a head or operand mix-up picks other dims)
    H, D_c, D_v, R = 3, 512, 128, 5
    o = wl.normal(31, "vc_o", R * H * D_c).reshape(R, H, D_c).astype(np.float32)
    sel = np.stack([(np.arange(D_v) * (2 * h + 3) + 7 * h + 1) % D_c for h in range(H)])
    w = np.zeros((H, D_c, D_v))
    for h in range(H):
        w[h, sel[h], np.arange(D_v)] = 1.0
    v = ot.vc_up_proj(o, _bf16_bits(w))
    for h in range(H):
        assert np.array_equal(v[:, h, :], o[:, h, sel[h]])


def test_vc_unit_latent_returns_weight_row():
    # o[r, h] = e_k: v[r, h] is row k of that head's weights (fixes which weight index
    # runs over the latent)
    H, D_c, D_v = 2, 512, 64
    w = _bf16_bits(wl.normal(32, "vc_w", H * D_c * D_v).reshape(H, D_c, D_v))
    wf = (w.astype(np.uint32) << np.uint32(16)).view(np.float32)
    ks = [0, 1, 255, 256, 511]
    o = np.zeros((len(ks), H, D_c), dtype=np.float32)
    for r, k in enumerate(ks):
        o[r, :, k] = 1.0
    v = ot.vc_up_proj(o, w)
    for r, k in enumerate(ks):
        for h in range(H):
            assert np.array_equal(v[r, h], wf[h, k])


def test_vc_triangular_closed_forms():
    # w[h, d, n] = 1 for d <= n: with o = 1 every output is n + 1; with o[d] = d it is
    # n (n + 1) / 2 -- closed forms that fix the summation range over the latent
    H, D_c, D_v = 2, 512, 256
    tri = (np.arange(D_c)[:, None] <= np.arange(D_v)[None, :]).astype(np.float64)
    w = _bf16_bits(np.broadcast_to(tri, (H, D_c, D_v)))
    n = np.arange(D_v, dtype=np.float64)
    v1 = ot.vc_up_proj(np.ones((2, H, D_c), dtype=np.float32), w)
    assert np.array_equal(v1, np.broadcast_to((n + 1).astype(np.float32), v1.shape))
    od = np.broadcast_to(np.arange(D_c, dtype=np.float32), (3, H, D_c))
    v2 = ot.vc_up_proj(od, w)
    assert np.array_equal(v2, np.broadcast_to((n * (n + 1) / 2).astype(np.float32), v2.shape))


def test_vc_bf16_weights_widen_exactly():
    # bit patterns with known values: 1, -2, 0.5 + 2^-8 (the last mantissa bit), the largest
    # finite bf16 and the smallest subnormal
    bits = np.array([0x3F80, 0xC000, 0x3F01, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -2.0, 0.50390625, (2 - 2 ** -7) * 2.0 ** 127, 2.0 ** -133]
    w = bits.reshape(1, 5, 1) * np.ones((1, 1, 1), dtype=np.uint16)
    for k in range(5):
        o = np.zeros((1, 1, 5), dtype=np.float32)
        o[0, 0, k] = 1.0
        assert float(ot.vc_up_proj(o, w)[0, 0, 0]) == np.float32(want[k])
