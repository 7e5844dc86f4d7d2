"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same
seeded inputs. Visibility bits must match bit for bit; attention must satisfy
|gpu - oracle| <= atol + rtol*|oracle| elementwise on out and lse with
(atol, rtol) = (1e-4, 1e-4) for fp32 inputs and (2e-2, 2e-2) for bf16 inputs."""
import zlib

import numpy as np
import pytest

import workloads as wl
from tests import gpu_util as G
from tests import helpers as H

pytestmark = pytest.mark.gpu

IMPLS_BY_DTYPE = {"f32": ["simt", "simt_small"], "bf16": ["simt", "simt_small", "tcgen05"]}


@pytest.fixture(scope="module")
def kdt():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_absorb_gb300 import build_lib
    build_lib.build()
    import speculative_decoding_tree_absorb_gb300 as k
    return k


def _compare(case, out, lse, ref_out, ref_lse, what):
    atol, rtol = H.TOL[case.dtype]
    H.assert_close(out, ref_out, atol, rtol, what + " out")
    H.assert_close(lse, ref_lse, atol, rtol, what + " lse")


# ---------------------------------------------------------------- visibility --

def test_visibility_bit_exact_on_every_small_tree(kdt, oracle_mod):
    import torch
    for T in range(1, 7):
        parents = np.stack(list(H.all_parent_arrays(T)))
        got = kdt.build_visibility(torch.from_numpy(parents).cuda()).cpu().numpy().view(np.uint32)
        np.testing.assert_array_equal(got, oracle_mod.build_visibility(parents))


@pytest.mark.parametrize("T", [1, 9, 31, 32, 33, 64, 100, 128, 129, 200, 1000])
@pytest.mark.parametrize("kind", ["uniform", "geometric", "depth16", "window8", "chain", "star"])
def test_visibility_bit_exact_on_config_trees(kdt, oracle_mod, T, kind):
    import torch
    parents = np.stack([wl.TREE_KINDS[kind](77, f"v/{b}", T) for b in range(5)])
    got = kdt.build_visibility(torch.from_numpy(parents).cuda()).cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, oracle_mod.build_visibility(parents))


def test_visibility_error_word_matches_oracle(kdt, oracle_mod):
    import torch
    p = np.stack([wl.tree_geometric(5, f"e/{b}", 40) for b in range(3)])
    p[2, 7] = 9            # >= i
    p[1, 30] = -3          # < -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kdt.build_visibility(torch.from_numpy(p).cuda(), err=err)
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_visibility(p)
    assert int(err.item()) == 1 * 40 + 30 + 1
    assert f"flat index {1 * 40 + 30}" in str(e.value)
    # a well-formed tree clears the word
    kdt.build_visibility(torch.from_numpy(p[:1].copy()).cuda(), err=err)
    assert int(err.item()) == 0


# ------------------------------------------------------------------- attention --

EDGE_CASES = [
    # name, B, T, H, prefix, tree
    ("pages_p0_b8", 2, 9, 8, 0, "uniform"),
    ("pages_p1_b4", 3, 5, 8, 1, "uniform"),
    ("pages_p37_b8", 2, 9, 8, 37, "uniform"),
    ("single_query", 2, 1, 8, 70, "uniform"),
    ("t31", 1, 31, 4, 19, "geometric"),
    ("t32", 2, 32, 2, 64, "uniform"),
    ("t33", 2, 33, 2, 63, "depth16"),
    ("ragged_tail", 3, 17, 4, (3, 130, 64), "geometric"),
    ("one_head", 2, 12, 1, (5, 200), "window8"),
    ("h16_multi_tile", 1, 20, 16, 150, "uniform"),
    ("chain", 2, 24, 8, 90, "chain"),
    ("star", 2, 24, 8, 90, "star"),
    ("h128", 1, 3, 128, 300, "uniform"),
    ("wide_tree", 1, 130, 2, 10, "geometric"),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name,B,T,Hh,prefix,tree", EDGE_CASES)
def test_edge_cases_match_oracle(kdt, oracle_mod, dtype, name, B, T, Hh, prefix, tree):
    case = wl.make_case(name, B=B, T=T, H=Hh, prefix=prefix, dtype=dtype, tree=tree, seed=zlib.crc32(name.encode()) % 1000)
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    for impl in IMPLS_BY_DTYPE[dtype]:
        for use_bits in (False, True):
            out, lse, err = G.run(case, impl=impl, use_bits=use_bits)
            assert err == 0
            assert np.isfinite(out).all() and np.isfinite(lse).all()
            _compare(case, out, lse, ref_out, ref_lse, f"{name}/{impl}/bits={use_bits}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiny_config_full(kdt, oracle_mod, dtype):
    case = wl.make_config("tiny", dtype=dtype)
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    for impl in IMPLS_BY_DTYPE[dtype]:
        out, lse, err = G.run(case, impl=impl)
        assert err == 0
        _compare(case, out, lse, ref_out, ref_lse, f"tiny/{impl}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_result_independent_of_split_count(kdt, oracle_mod, dtype):
    # SIMT 64-row tile: num_splits CTAs sharing the (row tile, key block) pairs; 16-row
    # tile: num_splits KV ranges per row tile, merged by the split-merge kernel. Tensor
    # path: num_splits persistent clusters sharing the (unit, key block) work. Every count
    # moves the boundaries that cut tiles or units into pieces (1 = no pieces at all).
    import torch
    case = wl.make_case("splits", B=3, T=16, H=8, prefix=(700, 33, 1000), dtype=dtype, tree="geometric", seed=5)
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    d = G.to_device(case)
    for impl in IMPLS_BY_DTYPE[dtype]:
        base = None
        for s in (1, 2, 3, 5, 8, 17, 32):
            out_t = torch.empty((case.B, case.T, case.H, 512), device="cuda")
            pl = kdt.plan(kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"],
                                        parent=d["parent"], max_kv_len=case.max_kv_len, out=out_t, impl=impl,
                                        num_splits=s))
            if impl == "tcgen05":
                assert pl["num_splits"] == s and pl["ctas"] == 4 * s
                assert pl["num_launches"] == (3 if s > 1 else 2)      # bits, attention (, piece merge)
            out, lse, _ = G.run(case, impl=impl, num_splits=s, dev_tensors=d)
            _compare(case, out, lse, ref_out, ref_lse, f"splits={s}/{impl}")
            if base is None:
                base = (out, lse)
            else:
                # SIMT keeps P in fp32, so splits agree to fp32 rounding; the tensor path
                # rounds P to bf16 relative to each split's running max, so two split
                # counts differ by up to that rounding and are held to the bf16 bound.
                atol, rtol = (1e-5, 1e-5) if impl == "simt" else H.TOL["bf16"]
                H.assert_close(out, base[0], atol, rtol, "split vs unsplit")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_caller_bits_including_empty_rows(kdt, oracle_mod, dtype):
    case = wl.make_case("bits", B=2, T=40, H=4, prefix=(0, 65), dtype=dtype, tree="uniform", seed=8)
    vis = wl.random_vis_bits(8, "bits", case.B, case.T, density=0.3, force_self=False)
    vis[0, 3] = 0            # prefix 0 and no bit: empty visible set
    vis[0, 39] = 0
    ref_out, ref_lse = oracle_mod.verify_attn(case, vis=vis)
    for impl in IMPLS_BY_DTYPE[dtype]:
        out, lse, _ = G.run(case, impl=impl, vis=vis)
        assert np.isneginf(lse[0, 3]).all() and (out[0, 3] == 0).all()
        _compare(case, out, lse, ref_out, ref_lse, f"bits/{impl}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_visible_key_is_exact(kdt, dtype):
    case = wl.make_case("one", B=2, T=6, H=64, prefix=0, dtype=dtype, tree="uniform", seed=13)
    for impl in IMPLS_BY_DTYPE[dtype]:
        out, lse, _ = G.run(case, impl=impl)
        want = H.widen(case.c_kv[:, 0], dtype)
        for h in range(case.H):
            np.testing.assert_array_equal(out[:, 0, h].astype(np.float64), want)


def test_golden_zero_query_closed_form(kdt):
    for dtype in ("f32", "bf16"):
        for g in H.read_golden_cases("q_zero_uniform.txt"):
            T = len(g["parent"])
            case = wl.make_case(g["name"], B=1, T=T, H=8, prefix=g["prefix"], dtype=dtype, tree=g["parent"], seed=5)
            case.q_nope[:] = 0
            case.q_pe[:] = 0
            for impl in IMPLS_BY_DTYPE[dtype]:
                out, lse, _ = G.run(case, impl=impl)
                np.testing.assert_allclose(lse[0], np.log(np.array(g["count"], dtype=np.float64))[:, None]
                                           * np.ones((1, 8)), rtol=1e-5, atol=1e-5)
                ck = H.widen(case.c_kv[0], dtype)
                for i, path in g["paths"].items():
                    rows = list(range(g["prefix"])) + [g["prefix"] + t for t in path]
                    np.testing.assert_allclose(out[0, i], np.broadcast_to(ck[rows].mean(0), (8, 512)),
                                               rtol=1e-4, atol=1e-5)


def test_merge_attn_states_matches_oracle(kdt, oracle_mod):
    import torch
    rng = np.random.default_rng(3)
    n, D = 1000, 512
    o_a = rng.standard_normal((n, D)).astype(np.float32)
    o_b = rng.standard_normal((n, D)).astype(np.float32)
    la = (rng.standard_normal(n) * 5).astype(np.float32)
    lb = (rng.standard_normal(n) * 5).astype(np.float32)
    la[::7] = -np.inf
    lb[::11] = -np.inf
    ref_o, ref_l = oracle_mod.merge_states(o_a, la, o_b, lb)
    t = [torch.from_numpy(x).cuda() for x in (o_a, la, o_b, lb)]
    o, l = kdt.merge_attn_states(*t)
    H.assert_close(o.cpu().numpy(), ref_o, 1e-5, 1e-5, "merge o")
    H.assert_close(l.cpu().numpy(), ref_l, 1e-5, 1e-5, "merge lse")
    # in place into the first state
    kdt.merge_attn_states(*t, out=t[0], lse=t[1])
    H.assert_close(t[0].cpu().numpy(), ref_o, 1e-5, 1e-5, "merge in place")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_running_max_jumps_force_output_rescale(kdt, oracle_mod, dtype):
    # The second half of every cache is scaled x6: scores jump well past the running
    # maximum set by the first blocks, so accumulated outputs must be rescaled.
    case = wl.make_case("jump", B=2, T=16, H=16, prefix=(1500, 900), dtype=dtype, tree="geometric", seed=3)
    for b in range(case.B):
        n = int(case.kv_len[b])
        if dtype == "bf16":
            x = wl.bf16_bits_to_f32(case.c_kv[b, n // 2:n]).astype(np.float64) * 6.0
            case.c_kv[b, n // 2:n] = wl.f64_to_bf16_bits(x)
        else:
            case.c_kv[b, n // 2:n] *= 6.0
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    # The absolute error of the output grows with the magnitude of the values it averages
    # (fp32: rounding of the 576-term score dots and the sums; bf16: rounding of P), and
    # the cache here is 6x larger than in the N(0,1) configurations, so the absolute
    # term of each bound is scaled by 6; the relative term is unchanged.
    atol, rtol = (6e-4, 1e-4) if dtype == "f32" else (6 * 2e-2, 2e-2)
    for impl in IMPLS_BY_DTYPE[dtype]:
        for s in (0, 1, 4):
            out, lse, err = G.run(case, impl=impl, num_splits=s)
            assert err == 0
            H.assert_close(out, ref_out, atol, rtol, f"jump/{impl}/splits={s} out")
            H.assert_close(lse, ref_lse, atol, rtol, f"jump/{impl}/splits={s} lse")


def test_tail_tiles_split_to_fill_the_last_wave(kdt, oracle_mod):
    # 2 sequences x 20 units of 256 rows, 6 key blocks each: one wave of whole units on the
    # resident clusters, then a tail of units cut into key ranges and merged afterwards.
    import torch
    case = wl.make_case("tail", B=2, T=40, H=128, prefix=(700, 650), dtype="bf16", tree="geometric", seed=17)
    d = G.to_device(case)
    out = torch.empty((case.B, case.T, case.H, 512), device="cuda")
    a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                      max_kv_len=case.max_kv_len, out=out)
    pl = kdt.plan(a)
    assert pl["impl"] == "tcgen05" and pl["num_launches"] == 3          # visibility, attention, tail merge
    out_g, lse_g, err = G.run(case, impl="auto", dev_tensors=d)
    assert err == 0
    rows_tail = np.arange(case.rows - 5 * 256, case.rows)               # the tail units and the last whole one
    rows = np.unique(np.concatenate([rows_tail, _sample_rows(case, 128, seed=4)]))
    ref_out, ref_lse = oracle_mod.verify_attn_rows(case, rows)
    _compare(case, out_g.reshape(-1, 512)[rows], lse_g.reshape(-1)[rows], ref_out, ref_lse, "tail")


def test_auto_picks_tensor_cores_for_bf16(kdt):
    import torch
    case = wl.make_case("plan", B=2, T=16, H=64, prefix=300, dtype="bf16", seed=1)
    d = G.to_device(case)
    out = torch.empty((case.B, case.T, case.H, 512), device="cuda")
    a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                      max_kv_len=case.max_kv_len, out=out)
    assert kdt.plan(a)["impl"] == "tcgen05"
    # small problems take the SIMT kernel on 16-row tiles, whatever the dtype; larger fp32
    # problems the SIMT kernel on 64-row tiles
    for dtype, prefix, want in (("f32", 30, "simt_small"), ("bf16", 30, "simt_small"), ("f32", 4000, "simt")):
        f = wl.make_case("plan32", B=1, T=16, H=64, prefix=prefix, dtype=dtype, seed=1)
        d = G.to_device(f)
        out = torch.empty((f.B, f.T, f.H, 512), device="cuda")
        a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                          max_kv_len=f.max_kv_len, out=out)
        assert kdt.plan(a)["impl"] == want, (dtype, prefix)


# ------------------------------------------------------- full-size configurations --

def _sample_rows(case, n, seed):
    rng = np.random.default_rng(seed)
    rows = rng.choice(case.rows, size=min(n, case.rows), replace=False)
    # always include the first and last row of every sequence (tile edges)
    edge = np.concatenate([[b * case.T * case.H, (b + 1) * case.T * case.H - 1] for b in range(case.B)])
    return np.unique(np.concatenate([rows, edge]))


@pytest.mark.parametrize("name", ["kimi", "ragged", "target", "long", "dsv3"])
def test_full_size_config_every_element(kdt, oracle_mod, name):
    # The launch configuration the bench times (automatic plan), every element of out and
    # lse against the oracle on all host cores (about 10-90 s of oracle time per workload).
    case = wl.make_config(name)
    out, lse, err = G.run(case, impl="auto")
    assert err == 0
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ref_out, ref_lse = oracle_mod.verify_attn(case)   # the bits passed for DSv3 are the tree's
    _compare(case, out, lse, ref_out, ref_lse, name)


def test_tensors_outside_device_memory_are_refused_before_any_launch(kdt):
    # Pinned host memory (reachable from the GPU through unified addressing) and pageable
    # host memory are refused with KDT_ERR_NOT_DEVICE: nothing runs, so the error word
    # keeps its sentinel and the output its NaNs.
    import ctypes
    import torch
    case = wl.make_case("where", B=2, T=8, H=64, prefix=200, dtype="bf16", tree="geometric", seed=21)
    d = G.to_device(case)
    K = kdt.kdt
    for impl in ("tcgen05", "simt"):
        for where in ("pinned", "pageable"):
            c_kv = d["c_kv"].cpu()
            if where == "pinned":
                c_kv = c_kv.pin_memory()
            out = torch.full((case.B, case.T, case.H, 512), float("nan"), device="cuda")
            err = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
            a = kdt.make_args(d["q_nope"], d["q_pe"], c_kv, d["k_pe"], d["prefix_len"], parent=d["parent"],
                              max_kv_len=case.max_kv_len, out=out, err=err, impl=impl)
            ws = torch.empty(max(1, kdt.workspace_size(a)), dtype=torch.uint8, device="cuda")
            st = kdt.lib().kdt_verify_attn(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
            torch.cuda.synchronize()
            assert st == K.KDT_ERR_NOT_DEVICE, (impl, where, st)
            assert int(err.item()) == 12345 and torch.isnan(out).all()
        # the same call with every tensor on the device runs
        out = torch.empty((case.B, case.T, case.H, 512), device="cuda")
        a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                          max_kv_len=case.max_kv_len, out=out, impl=impl)
        ws = torch.empty(max(1, kdt.workspace_size(a)), dtype=torch.uint8, device="cuda")
        assert kdt.lib().kdt_verify_attn(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), ws.numel(), None) == K.KDT_OK
        # a workspace in host memory is refused too
        wsh = torch.empty(max(1, kdt.workspace_size(a)), dtype=torch.uint8).pin_memory()
        assert kdt.lib().kdt_verify_attn(ctypes.byref(a), ctypes.c_void_p(wsh.data_ptr()), wsh.numel(),
                                         None) == K.KDT_ERR_NOT_DEVICE
    torch.cuda.synchronize()
