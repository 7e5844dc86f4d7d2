"""GPU parity for the steps next to verify: NeoX RoPE, greedy tree accept and cache
compaction, through the C ABI, against the CPU oracle (oracle/tree_ops.py) on the same
seeded inputs.

Bars: accept, compaction and the tree builder are integer, copy and float32-sum work --
bit-exact. RoPE takes its angles in float64 and rounds their cosines and sines to
float32 on both sides, then does the same float32 operations; the two sides may differ
only where the float64 cosine or sine of the GPU's math library and of the host's differ
in the last bit and straddle a float32 rounding boundary, so the bar is at most one unit
in the last place of the element type, with every element that is not rotated
bit-exact.
"""
import numpy as np
import pytest

import workloads as wl
from oracle import tree_ops as ot

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kdt():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_absorb_gb300 import build_lib
    build_lib.build()
    import speculative_decoding_tree_absorb_gb300 as k
    return k


def _stored(seed, tag, shape, dtype):
    """Seeded N(0,1) values as stored: float32 array, or bf16 bit patterns (uint16)."""
    x = wl.normal(seed, tag, int(np.prod(shape))).reshape(shape)
    return x.astype(np.float32) if dtype == "f32" else wl.f64_to_bf16_bits(x)


def _widen(a, dtype):
    return a.astype(np.float32) if dtype == "f32" else wl.bf16_bits_to_f32(a).astype(np.float32)


def _round(x, dtype):
    """float32 oracle values to the element type as stored (bf16: round to nearest even)."""
    return x.astype(np.float32) if dtype == "f32" else wl.f64_to_bf16_bits(x.astype(np.float64))


def _to_dev(a, dtype):
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _from_dev(t, dtype):
    import torch
    if dtype == "f32":
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _ulp_diff(a, b, dtype):
    """Distance in units in the last place between same-typed stored values."""
    if dtype == "f32":
        ia = a.view(np.int32).astype(np.int64)
        ib = b.view(np.int32).astype(np.int64)
        ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
        ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    else:
        ia = a.astype(np.int64)
        ib = b.astype(np.int64)
        ia = np.where(ia >= 0x8000, -(ia & 0x7FFF), ia)
        ib = np.where(ib >= 0x8000, -(ib & 0x7FFF), ib)
    return np.abs(ia - ib)


# ---------------------------------------------------------------------- RoPE --
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,H,prefix", [(1, 1, 1, 0), (3, 20, 8, 100), (2, 64, 64, 8192)])
def test_rope_in_place_on_combined_query_and_tree_keys(kdt, dtype, B, T, H, prefix):
    import torch
    L = prefix + T + 5
    q_comb = _stored(1, "qc", (B, T, H, 576), dtype)
    k_pe = _stored(2, "kp", (B, L, 64), dtype)
    pre = np.array([prefix - 3 * b if prefix >= 3 * b else 0 for b in range(B)], dtype=np.int32)
    par = np.stack([wl.tree_geometric(b, "rope", T) for b in range(B)])
    pos = ot.tree_positions(par, pre).astype(np.int32)
    base = 10000.0
    dq, dk = _to_dev(q_comb, dtype), _to_dev(k_pe, dtype)
    kdt.rope_neox(torch.from_numpy(pos).cuda(), q=dq[..., 512:], k_pe=dk,
                  prefix_len=torch.from_numpy(pre).cuda(), base=base)
    torch.cuda.synchronize()
    gq, gk = _from_dev(dq, dtype), _from_dev(dk, dtype)
    # the nope part of every query row is untouched
    assert np.array_equal(gq[..., :512], q_comb[..., :512])
    ref_q = _round(ot.rope_neox(_widen(q_comb[..., 512:], dtype), pos[:, :, None], base), dtype)
    d = _ulp_diff(gq[..., 512:], ref_q, dtype)
    assert d.max() <= 1, f"rope q: {int((d > 0).sum())} elements differ, max {int(d.max())} ulp"
    # key rows prefix + i rotated by pos[b, i]; every other row untouched
    ref_k = k_pe.copy()
    for b in range(B):
        rows = pre[b] + np.arange(T)
        ref_k[b, rows] = _round(ot.rope_neox(_widen(k_pe[b, rows], dtype), pos[b], base), dtype)
    d = _ulp_diff(gk, ref_k, dtype)
    assert d.max() <= 1, f"rope k: {int((d > 0).sum())} elements differ"
    untouched = np.ones((B, L), dtype=bool)
    for b in range(B):
        untouched[b, pre[b]:pre[b] + T] = False
    assert np.array_equal(gk[untouched], k_pe[untouched])


def test_rope_position_zero_is_exact_identity(kdt):
    import torch
    q = _stored(3, "q0", (2, 4, 3, 64), "f32")
    dq = _to_dev(q, "f32")
    kdt.rope_neox(torch.zeros((2, 4), dtype=torch.int32, device="cuda"), q=dq, base=10000.0)
    assert np.array_equal(_from_dev(dq, "f32"), q)


# -------------------------------------------------------------------- accept --
def _accept_inputs(seed, B, T):
    par = np.stack([(wl.tree_uniform(seed + b, "acc", T) if (seed + b) % 2 else wl.tree_geometric(seed + b, "acc", T))
                    for b in range(B)]).astype(np.int32)
    tok = (wl.raw_u64(seed, "tok", B * T) % 3).astype(np.int32).reshape(B, T)    # repeats: ties happen
    tgt = (wl.raw_u64(seed, "tgt", B * T) % 3).astype(np.int32).reshape(B, T)
    return par, tok, tgt


@pytest.mark.parametrize("B,T", [(1, 1), (4, 5), (16, 64), (8, 300), (2, 4096)])
def test_accept_bit_exact(kdt, B, T):
    import torch
    par, tok, tgt = _accept_inputs(T, B, T)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, n, bonus = kdt.tree_accept(*(torch.from_numpy(a).cuda() for a in (par, tok, tgt)), err=err)
    acc, n, bonus = acc.cpu().numpy(), n.cpu().numpy(), bonus.cpu().numpy()
    assert int(err.item()) == 0
    for b, (path, bon) in enumerate(ot.tree_accept(par, tok, tgt)):
        assert n[b] == len(path) and bonus[b] == bon
        assert acc[b, :len(path)].tolist() == path and (acc[b, len(path):] == -1).all()


def test_accept_chain_all_match_and_malformed_entry(kdt):
    import torch
    T = 64
    par = wl.tree_chain(T)[None].astype(np.int32)
    tgt = (np.arange(T) + 7)[None].astype(np.int32)
    tok = np.concatenate([[0], tgt[0, :-1]])[None].astype(np.int32)
    acc, n, bonus = kdt.tree_accept(*(torch.from_numpy(a).cuda() for a in (par, tok, tgt)))
    assert int(n.item()) == T and acc.cpu().numpy()[0].tolist() == list(range(T)) and int(bonus.item()) == tgt[0, -1]
    bad = par.copy()
    bad[0, 10] = 12                                     # points forward: malformed
    bad[0, 20] = -5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, n, bonus = kdt.tree_accept(*(torch.from_numpy(a).cuda() for a in (bad, tok, tgt)), err=err)
    assert int(err.item()) == 1 + 10
    assert int(n.item()) == 10                          # the walk stops where the chain was cut


# ---------------------------------------------------------------- compaction --
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,prefix", [(1, 1, 0), (4, 16, 37), (8, 64, 8192)])
def test_compact_bit_exact_with_prefix_update(kdt, dtype, B, T, prefix):
    import torch
    L = prefix + T + 3
    c = _stored(5, "ckv", (B, L, 512), dtype)
    k = _stored(6, "kpe", (B, L, 64), dtype)
    pre = np.array([max(prefix - b, 0) for b in range(B)], dtype=np.int32)
    # a deep accepted path: chain-heavy trees and targets that match most drafts
    par = np.stack([wl.tree_geometric(b, "cmp", T, q=0.8) for b in range(B)]).astype(np.int32)
    tgt = (wl.raw_u64(9, "t", B * T) % 2).astype(np.int32).reshape(B, T)
    tok = np.zeros((B, T), dtype=np.int32)
    for b in range(B):
        for i in range(1, T):
            tok[b, i] = tgt[b, par[b, i]] if (i % 5) else 1 - tgt[b, par[b, i]]
    d_par, d_tok, d_tgt = (torch.from_numpy(a).cuda() for a in (par, tok, tgt))
    acc, n, _ = kdt.tree_accept(d_par, d_tok, d_tgt)
    dc, dk, dpre = _to_dev(c, dtype), _to_dev(k, dtype), torch.from_numpy(pre).cuda()
    kdt.kv_compact(dc, dk, dpre, acc, n)
    torch.cuda.synchronize()
    paths = [p for p, _ in ot.tree_accept(par, tok, tgt)]
    rc, rk, rp = ot.kv_compact(c, k, pre, paths)
    assert np.array_equal(_from_dev(dc, dtype), rc)
    assert np.array_equal(_from_dev(dk, dtype), rk)
    assert dpre.cpu().numpy().tolist() == rp.tolist()


# ------------------------------------- verify reading the combined query buffer --
@pytest.mark.parametrize("dtype,impl", [("f32", "simt"), ("bf16", "simt"), ("bf16", "tcgen05")])
def test_verify_reads_combined_query_buffer_bit_for_bit(kdt, dtype, impl):
    import torch
    from tests import gpu_util as G
    case = wl.make_case("comb", B=2, T=16, H=64, prefix=(700, 300), dtype=dtype, tree="geometric", seed=5)
    d = G.to_device(case)
    comb = torch.cat([d["q_nope"], d["q_pe"]], dim=-1).contiguous()      # [B,T,H,576]
    kw = dict(parent=d["parent"], scale=case.scale, impl=impl, max_kv_len=case.max_kv_len)
    out_a, lse_a = kdt.verify_attn(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], **kw)
    out_b, lse_b = kdt.verify_attn(comb[..., :512], comb[..., 512:], d["c_kv"], d["k_pe"], d["prefix_len"], **kw)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


def test_device_chain_rope_verify_accept_compact(kdt, oracle_mod):
    """One DDTree step on the device with no host round trip between the steps: rotate the
    combined query buffer and the tree's key rows, verify from the combined buffer, accept
    greedily on seeded synthetic target tokens, compact the rotated cache. The oracle runs
    the same chain on the same seeded inputs with its own results at every step."""
    import dataclasses

    import torch
    from tests import gpu_util as G
    from tests import helpers as H
    case = wl.make_case("chain", B=3, T=24, H=16, prefix=(900, 400, 1500), dtype="bf16", tree="geometric", seed=8)
    d = G.to_device(case)
    B, T, Hh = case.B, case.T, case.H
    comb = torch.cat([d["q_nope"], d["q_pe"]], dim=-1).contiguous()
    pos_h = ot.tree_positions(case.parent, case.prefix_len).astype(np.int32)
    tok_h = (wl.raw_u64(8, "tok", B * T) % 2).astype(np.int32).reshape(B, T)
    tgt_h = (wl.raw_u64(8, "tgt", B * T) % 2).astype(np.int32).reshape(B, T)
    pos, tok, tgt = (torch.from_numpy(a).cuda() for a in (pos_h, tok_h, tgt_h))
    # -- device chain
    kdt.rope_neox(pos, q=comb[..., 512:], k_pe=d["k_pe"], prefix_len=d["prefix_len"], base=10000.0)
    out, lse = kdt.verify_attn(comb[..., :512], comb[..., 512:], d["c_kv"], d["k_pe"], d["prefix_len"],
                               parent=d["parent"], scale=case.scale, max_kv_len=case.max_kv_len)
    acc, n_acc, bonus = kdt.tree_accept(d["parent"], tok, tgt)
    kdt.kv_compact(d["c_kv"], d["k_pe"], d["prefix_len"], acc, n_acc)
    torch.cuda.synchronize()
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    # -- the oracle's chain
    r_qpe = _round(ot.rope_neox(_widen(case.q_pe, "bf16"), pos_h[:, :, None], 10000.0), "bf16")
    r_kpe = case.k_pe.copy()
    for b in range(B):
        rr = case.prefix_len[b] + np.arange(T)
        r_kpe[b, rr] = _round(ot.rope_neox(_widen(case.k_pe[b, rr], "bf16"), pos_h[b], 10000.0), "bf16")
    assert _ulp_diff(bits(comb[..., 512:]), r_qpe, "bf16").max() <= 1
    rows = np.arange(B * T * Hh)[::7]
    ref_o, ref_l = oracle_mod.verify_attn_rows(dataclasses.replace(case, q_pe=r_qpe, k_pe=r_kpe), rows)
    H.assert_close(out.reshape(-1, 512)[rows].cpu().numpy(), ref_o, *H.TOL["bf16"], "chain out")
    H.assert_close(lse.reshape(-1)[rows].cpu().numpy(), ref_l, *H.TOL["bf16"], "chain lse")
    res = ot.tree_accept(case.parent, tok_h, tgt_h)
    assert n_acc.cpu().numpy().tolist() == [len(p) for p, _ in res]
    assert bonus.cpu().numpy().tolist() == [bn for _, bn in res]
    rc, rk, rp = ot.kv_compact(case.c_kv, r_kpe, case.prefix_len, [p for p, _ in res])
    assert np.array_equal(bits(d["c_kv"]), rc)
    assert _ulp_diff(bits(d["k_pe"]), rk, "bf16").max() <= 1
    assert d["prefix_len"].cpu().numpy().tolist() == rp.tolist()
    assert sum(len(p) for p, _ in res) > B                                  # some draft token was accepted


# ------------------------------------------------------------------ builder --
def _cand(seed, B, D, K, quant):
    lp = -np.abs(wl.normal(seed, "blp", B * D * K)).reshape(B, D, K)
    if quant:                                            # ties in scores and within a depth
        lp = -np.round(-lp * 2.0) / 2.0
    tok = (wl.raw_u64(seed, "btok", B * D * K) % 50000).astype(np.int32).reshape(B, D, K)
    return tok, lp.astype(np.float32)


# N + 1 <= 32, 64, 128 take the register-resident kernel (one, two, four slots a lane),
# larger trees the shared-memory one; the cases sit on both sides of each boundary, and
# (3, 2, 5, 30) and (2, 1, 32, 32) use up every candidate.
@pytest.mark.parametrize("B,D,K,N,quant", [(4, 8, 4, 63, False), (2, 16, 8, 255, False), (3, 4, 3, 60, True),
                                           (2, 5, 1, 5, False), (2, 3, 3, 39, True), (1, 64, 32, 4095, False),
                                           (5, 12, 6, 127, True), (2, 6, 2, 31, False), (2, 7, 3, 64, True),
                                           (2, 9, 2, 128, False), (3, 2, 5, 30, False), (2, 1, 32, 32, True)])
def test_build_bit_exact(kdt, B, D, K, N, quant):
    import torch
    tok, lp = _cand(D * 100 + K, B, D, K, quant)
    root = np.arange(B, dtype=np.int32) + 11
    g = kdt.tree_build(torch.from_numpy(tok).cuda(), torch.from_numpy(lp).cuda(), N,
                       root_tok=torch.from_numpy(root).cuda())
    g = [t.cpu().numpy() for t in g]
    r = ot.tree_build(tok, lp, N, root_tok=root)
    for name, a, e in zip(("parent", "tok", "depth", "score"), g, r):
        assert np.array_equal(a, e), f"{name} differs at {np.argwhere(a != e)[:5].tolist()}"


def test_device_step_from_builder(kdt, oracle_mod):
    """Build the tree from synthetic drafter candidates, then visibility, positions, RoPE,
    verify from the combined query buffer, accept and compaction, all queued on the device
    before one synchronisation; the oracle runs the same step on the same inputs."""
    import dataclasses

    import torch
    from tests import gpu_util as G
    from tests import helpers as H
    B, D, K, N, Hh = 3, 8, 4, 47, 16
    T = N + 1
    case = wl.make_case("step", B=B, T=T, H=Hh, prefix=(600, 1200, 333), dtype="bf16", tree="chain", seed=21)
    ctok, clp = _cand(21, B, D, K, False)
    tgt_h = (wl.raw_u64(21, "tgt", B * T) % 50000).astype(np.int32).reshape(B, T)
    # the oracle's tree; targets agree with the draft on a few nodes so some are accepted
    r_par, r_tok, r_dep, _ = ot.tree_build(ctok, clp, N)
    for b in range(B):
        for i in range(1, T):
            if i % 3 == 1:
                tgt_h[b, r_par[b, i]] = r_tok[b, i]
    d = G.to_device(case)
    comb = torch.cat([d["q_nope"], d["q_pe"]], dim=-1).contiguous()
    # -- device
    par, tok, dep, _ = kdt.tree_build(torch.from_numpy(ctok).cuda(), torch.from_numpy(clp).cuda(), N)
    pos = (d["prefix_len"][:, None] + dep).to(torch.int32)
    kdt.rope_neox(pos, q=comb[..., 512:], k_pe=d["k_pe"], prefix_len=d["prefix_len"], base=10000.0)
    vis = kdt.build_visibility(par)
    out, lse = kdt.verify_attn(comb[..., :512], comb[..., 512:], d["c_kv"], d["k_pe"], d["prefix_len"], vis=vis,
                               scale=case.scale, max_kv_len=case.max_kv_len)
    acc, n_acc, bonus = kdt.tree_accept(par, tok, torch.from_numpy(tgt_h).cuda())
    kdt.kv_compact(d["c_kv"], d["k_pe"], d["prefix_len"], acc, n_acc)
    torch.cuda.synchronize()
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    # -- oracle
    assert np.array_equal(par.cpu().numpy(), r_par) and np.array_equal(tok.cpu().numpy(), r_tok)
    pos_h = ot.tree_positions(r_par, case.prefix_len)
    assert np.array_equal(pos.cpu().numpy(), pos_h)
    r_qpe = _round(ot.rope_neox(_widen(case.q_pe, "bf16"), pos_h[:, :, None], 10000.0), "bf16")
    r_kpe = case.k_pe.copy()
    for b in range(B):
        rr = case.prefix_len[b] + np.arange(T)
        r_kpe[b, rr] = _round(ot.rope_neox(_widen(case.k_pe[b, rr], "bf16"), pos_h[b], 10000.0), "bf16")
    rows = np.arange(B * T * Hh)[::5]
    rcase = dataclasses.replace(case, q_pe=r_qpe, k_pe=r_kpe, parent=r_par)
    ref_o, ref_l = oracle_mod.verify_attn_rows(rcase, rows)
    H.assert_close(out.reshape(-1, 512)[rows].cpu().numpy(), ref_o, *H.TOL["bf16"], "step out")
    H.assert_close(lse.reshape(-1)[rows].cpu().numpy(), ref_l, *H.TOL["bf16"], "step lse")
    res = ot.tree_accept(r_par, r_tok, tgt_h)
    assert n_acc.cpu().numpy().tolist() == [len(p) for p, _ in res]
    assert bonus.cpu().numpy().tolist() == [bn for _, bn in res]
    assert max(len(p) for p, _ in res) > 1
    rc, rk, rp = ot.kv_compact(case.c_kv, r_kpe, case.prefix_len, [p for p, _ in res])
    assert np.array_equal(bits(d["c_kv"]), rc)
    assert _ulp_diff(bits(d["k_pe"]), rk, "bf16").max() <= 1
    assert d["prefix_len"].cpu().numpy().tolist() == rp.tolist()


def test_rope_unaligned_rows_take_the_scalar_path(kdt):
    # rows whose rope part does not start on a 16-byte boundary are rotated one pair a thread
    import torch
    B, T, H, d = 2, 5, 3, 64
    buf = _stored(13, "qu", (B, T, H, d + 2), "bf16")
    dq = _to_dev(buf, "bf16")
    pos = (np.arange(B * T, dtype=np.int32).reshape(B, T) * 13 + 1)
    kdt.rope_neox(torch.from_numpy(pos).cuda(), q=dq[..., 1:1 + d], base=10000.0)
    g = _from_dev(dq, "bf16")
    ref = _round(ot.rope_neox(_widen(buf[..., 1:1 + d], "bf16"), pos[:, :, None], 10000.0), "bf16")
    assert _ulp_diff(g[..., 1:1 + d], ref, "bf16").max() <= 1
    assert np.array_equal(g[..., 0], buf[..., 0]) and np.array_equal(g[..., 1 + d], buf[..., 1 + d])
