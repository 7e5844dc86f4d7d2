"""kdt_verify_attn_host (host buffers, chunked copies pipelined with the compute) against
the oracle, on the same seeded inputs as the device-entry parity tests."""
from __future__ import annotations

import numpy as np
import pytest

import workloads as wl
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


def _host(case, pin=True):
    import torch

    def conv(x):                       # bf16 arrays arrive as uint16 bit patterns; int32 stays int32
        t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if x.dtype == np.uint16 else torch.from_numpy(x)
        t = t.contiguous()
        return t.pin_memory() if pin else t

    return dict(q_nope=conv(case.q_nope), q_pe=conv(case.q_pe), c_kv=conv(case.c_kv), k_pe=conv(case.k_pe),
                prefix_len=conv(case.prefix_len.astype(np.int32)), parent=conv(case.parent.astype(np.int32)))


def _run(kdt, case, n_chunks, *, bits=False, pin=True, impl="auto"):
    import torch
    h = _host(case, pin)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = {}
    if bits:
        kw["vis"] = kdt.build_visibility(h["parent"].cuda()).cpu()
        kw["vis"] = kw["vis"].pin_memory() if pin else kw["vis"]
    else:
        kw["parent"] = h["parent"]
    out, lse = kdt.verify_attn_host(h["q_nope"], h["q_pe"], h["c_kv"], h["k_pe"], h["prefix_len"], err=err,
                                    scale=case.scale, max_kv_len=case.max_kv_len, n_chunks=n_chunks, impl=impl, **kw)
    torch.cuda.synchronize()
    return out.numpy(), lse.numpy(), int(err.item())


CASES = [
    # name, B, T, H, prefix, tree, dtype
    ("host_tiny_f32", 2, 9, 8, 37, "uniform", "f32"),
    ("host_bf16_ragged", 4, 16, 64, (300, 517, 64, 1000), "geometric", "bf16"),
    ("host_bf16_b6", 6, 33, 8, (5, 129, 700, 64, 1, 260), "depth16", "bf16"),
]


@pytest.mark.parametrize("name,B,T,Hh,prefix,tree,dtype", CASES)
def test_host_entry_matches_oracle_for_every_chunking(kdt, oracle_mod, name, B, T, Hh, prefix, tree, dtype):
    case = wl.make_case(name, B=B, T=T, H=Hh, prefix=prefix, dtype=dtype, tree=tree, seed=len(name) * 7)
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    atol, rtol = H.TOL[case.dtype]
    chunkings = sorted({0, 1, B} | {c for c in (2, 3) if B % c == 0})
    for n in chunkings:
        for bits in (False, True):
            out, lse, err = _run(kdt, case, n, bits=bits)
            assert err == 0
            H.assert_close(out, ref_out, atol, rtol, f"{name}/chunks={n}/bits={bits} out")
            H.assert_close(lse, ref_lse, atol, rtol, f"{name}/chunks={n}/bits={bits} lse")


def test_host_entry_pageable_buffers(kdt, oracle_mod):
    """Pageable host memory gives the same results (the copies then serialise)."""
    case = wl.make_case("host_pageable", B=2, T=12, H=16, prefix=(40, 90), dtype="bf16", tree="geometric", seed=5)
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    out, lse, err = _run(kdt, case, 2, pin=False)
    assert err == 0
    H.assert_close(out, ref_out, *H.TOL["bf16"], "pageable out")
    H.assert_close(lse, ref_lse, *H.TOL["bf16"], "pageable lse")


def test_host_entry_error_word_is_global(kdt, oracle_mod):
    """A malformed parent entry in a later chunk is reported by its flat index over the whole
    batch, as by kdt_build_visibility on the whole batch (and the oracle)."""
    import torch
    case = wl.make_case("host_err", B=4, T=10, H=8, prefix=(20, 30, 40, 50), dtype="f32", tree="uniform", seed=9)
    case.parent[2, 6] = 8                    # >= i: sequence 2 sits in chunk 1 of 2 and chunk 2 of 4
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.build_visibility(case.parent)
    assert f"flat index {2 * 10 + 6}" in str(e.value)
    for n in (1, 2, 4):
        _, _, err = _run(kdt, case, n)
        assert err == 1 + 2 * 10 + 6, n
    full = torch.zeros(1, dtype=torch.int32, device="cuda")
    kdt.build_visibility(torch.from_numpy(case.parent.astype(np.int32)).cuda(), err=full)
    assert int(full.item()) == 1 + 2 * 10 + 6
