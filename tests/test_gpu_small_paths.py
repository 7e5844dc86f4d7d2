"""GPU: the one-pass small-shape kernel (every sequence within one 64-key block, the
visibility built in the kernel from the parent array) and the 64-row SIMT tile's work
split (CTAs sharing all (row tile, key block) pairs, pieces merged by log-sum-exp),
against the oracle on the same seeded inputs, with the tolerances of the parity tests:
(1e-4, 1e-4) for fp32 inputs and (2e-2, 2e-2) for bf16."""
import numpy as np
import pytest

import workloads as wl
from tests import gpu_util as G
from tests import helpers as H

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


def _compare(case, out, lse, ref_out, ref_lse, what):
    atol, rtol = H.TOL[case.dtype]
    H.assert_close(out, ref_out, atol, rtol, what + " out")
    H.assert_close(lse, ref_lse, atol, rtol, what + " lse")


def _plan(kdt, case, d, **kw):
    import torch
    out = torch.empty((case.B, case.T, case.H, 512), device="cuda")
    return kdt.plan(kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                                  max_kv_len=case.max_kv_len, out=out, **kw))


ONE_PASS_CASES = [
    # name, B, T, H, prefix, tree: rows not a multiple of 4, no prefix, a full 64-key block
    ("op_odd_rows", 3, 5, 3, (0, 7, 59), "uniform"),
    ("op_full_block_chain", 2, 64, 1, 0, "chain"),
    ("op_kv64", 2, 9, 5, 55, "geometric"),
    ("op_one_query", 4, 1, 7, (0, 1, 30, 63), "uniform"),
    # 17, 33, 48 and 49 keys: the kernel computes 32, 48, 48 and 64 keys (4, 6, 6 and 8
    # groups of 8, a compile-time count per sequence), the extra ones masked
    ("op_key_groups", 4, 7, 3, (10, 26, 41, 42), "geometric"),
    # more rows than one-row CTAs fit at once (one fp32 CTA an SM, two bf16): rows a CTA
    # fp32 / bf16 = 2 / 1, 4 / 2, 4 / 4 and 4 / 4 with a last CTA of fewer rows
    ("op_rows2", 2, 9, 16, 37, "uniform"),
    ("op_rows_mid", 4, 9, 16, 12, "chain"),
    ("op_rows4", 8, 9, 16, 50, "uniform"),
    ("op_rows4_ragged", 4, 9, 17, (20, 0, 55, 33), "geometric"),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name,B,T,Hh,prefix,tree", ONE_PASS_CASES)
def test_one_pass_kernel_matches_oracle(kdt, oracle_mod, dtype, name, B, T, Hh, prefix, tree):
    case = wl.make_case(name, B=B, T=T, H=Hh, prefix=prefix, dtype=dtype, tree=tree, seed=17)
    assert case.max_kv_len <= 64
    d = G.to_device(case)
    pl = _plan(kdt, case, d, impl="simt_small")
    assert pl["impl"] == "simt_small" and pl["num_launches"] == 1 and pl["workspace_bytes"] == 0
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    for use_bits in (False, True):
        out, lse, err = G.run(case, impl="simt_small", use_bits=use_bits, dev_tensors=d)
        assert err == 0
        _compare(case, out, lse, ref_out, ref_lse, f"{name}/bits={use_bits}")


@pytest.mark.parametrize("B,T", [(3, 20), (24, 50)])
def test_one_pass_error_word(kdt, oracle_mod, B, T):
    """The first malformed parent entry over the batch, as kdt_build_visibility reports it:
    written by one CTA for a small batch (B*T <= 1024), else by each sequence's first CTA
    into a word cleared before the launch; a well-formed tree then reports 0."""
    import torch
    prefix = 64 - T
    case = wl.make_case("op_err", B=B, T=T, H=4, prefix=prefix, dtype="f32", tree="geometric", seed=23)
    p = case.parent.copy()
    p[B - 1, T - 3] = T - 3          # >= i
    p[1, T // 2] = -3                # < -1
    expected = 1 + min((B - 1) * T + T - 3, 1 * T + T // 2)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.build_visibility(p)
    d = G.to_device(case)
    err = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    kdt.verify_attn(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=torch.from_numpy(p).cuda(),
                    err=err, scale=case.scale, impl="simt_small", max_kv_len=case.max_kv_len)
    torch.cuda.synchronize()
    assert int(err.item()) == expected
    out, lse, err2 = G.run(case, impl="simt_small", dev_tensors=d)
    assert err2 == 0


def test_one_pass_reads_combined_query_buffer_bit_for_bit(kdt):
    """Query rows inside a combined [B,T,H,576] buffer (row stride 576) take one copy per
    row instead of one per range: the same result bit for bit."""
    import torch
    case = wl.make_case("op_comb", B=2, T=9, H=8, prefix=37, dtype="f32", tree="uniform", seed=29)
    d = G.to_device(case)
    comb = torch.cat([d["q_nope"], d["q_pe"]], dim=-1).contiguous()
    kw = dict(parent=d["parent"], scale=case.scale, impl="simt_small", max_kv_len=case.max_kv_len)
    out_a, lse_a = kdt.verify_attn(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], **kw)
    out_b, lse_b = kdt.verify_attn(comb[..., :512], comb[..., 512:], d["c_kv"], d["k_pe"], d["prefix_len"], **kw)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("ctas", [1, 2, 7, 31, 152, 1000])
def test_simt_work_split_over_ragged_sequences(kdt, oracle_mod, ctas):
    """Equal shares of the (64-row tile, 128-key block) pairs of sequences of very
    different lengths (one of them a single block, one with no prefix): share boundaries
    fall inside tiles and across sequences, some CTAs get two pieces, and with more CTAs
    than pairs some get none."""
    case = wl.make_case("split_ragged", B=6, T=8, H=16, prefix=(0, 100, 257, 1000, 31, 600), dtype="f32",
                        tree="uniform", seed=11)
    d = G.to_device(case)
    pl = _plan(kdt, case, d, impl="simt", num_splits=ctas)
    pairs = 6 * 2 * ((1008 + 127) // 128)
    assert pl["impl"] == "simt" and pl["num_splits"] == min(ctas, pairs)
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    out, lse, err = G.run(case, impl="simt", num_splits=ctas, dev_tensors=d)
    assert err == 0
    _compare(case, out, lse, ref_out, ref_lse, f"ctas={ctas}")
