"""kdt_verify_attn_noalloc against kdt_verify_attn and the oracle, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device memory
when they call the library (for example a serving engine that reserved nearly all
HBM for its KV-cache pool at start-up, or a plugin that may not use its host's
allocator). It keeps its scratch in a fixed array inside libkdt.so, shared by all
calls on a device. This file is collected last so that a failure here leaves every
other test already run; it passes alone in a fresh process as well.

Two calls in a row with different shapes and data check that what the first call
left in the shared scratch cannot leak into the second.
"""
import ctypes

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


def _both(kdt, case, impl, num_splits=0):
    """Run the case through kdt_verify_attn and kdt_verify_attn_noalloc (parent input)."""
    import torch
    d = G.to_device(case)
    ref_out, ref_lse, _ = G.run(case, impl=impl, num_splits=num_splits, use_bits=False, dev_tensors=d)
    out = torch.full((case.B, case.T, case.H, 512), float("nan"), device="cuda")
    lse = torch.full((case.B, case.T, case.H), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kdt.verify_attn_noalloc(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], out=out, lse=lse,
                            parent=d["parent"], max_kv_len=case.max_kv_len, scale=case.scale, err=err,
                            impl=impl, num_splits=num_splits)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return (out.cpu().numpy(), lse.cpu().numpy()), (ref_out, ref_lse)


def _check(case, got, ref, oracle_mod=None):
    """got against the workspace entry point's result and, given the oracle, against it too."""
    atol, rtol = H.TOL[case.dtype]
    H.assert_close(got[0], ref[0], atol, rtol, f"{case.name} out")
    H.assert_close(got[1], ref[1], atol, rtol, f"{case.name} lse")
    if oracle_mod is not None:
        o_out, o_lse = oracle_mod.verify_attn(case)
        H.assert_close(got[0], o_out, atol, rtol, f"{case.name} out vs oracle")
        H.assert_close(got[1], o_lse, atol, rtol, f"{case.name} lse vs oracle")


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(kdt, oracle_mod):
    # call 1: fp32, one sequence, several KV splits -> partials and bits in the scratch
    a = wl.make_case("noalloc_a", B=1, T=32, H=64, prefix=1500, dtype="f32", tree="window8", seed=41)
    got, ref = _both(kdt, a, impl="simt", num_splits=3)
    _check(a, got, ref, oracle_mod)
    # call 2: bf16, ragged batch, different tree and split count reusing the same scratch
    b = wl.make_case("noalloc_b", B=3, T=20, H=16, prefix=(900, 31, 400), dtype="bf16", tree="geometric",
                     seed=42)
    got, ref = _both(kdt, b, impl="auto", num_splits=3)
    _check(b, got, ref, oracle_mod)


def _auto_simt_plan_over_limit(kdt):
    """A fp32 shape whose automatic split count on the 16-row SIMT tile (one split per 64-key
    block, each with a partial state of every row) needs more than the fixed scratch. (The
    64-row tile's pieces, two of 64 rows per CTA, always fit.)"""
    import torch
    for B in range(3, 12):
        c = wl.make_case("noalloc_simt", B=B, T=59, H=64, prefix=640, dtype="f32", tree="uniform", seed=44)
        d = G.to_device(c)
        out = torch.empty((c.B, c.T, c.H, 512), device="cuda")
        a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                          max_kv_len=c.max_kv_len, scale=c.scale, out=out, impl="simt_small")
        if kdt.workspace_size(a) > (64 << 20):
            return c, kdt.plan(a)
    return None, None


def test_noalloc_fits_automatic_splits_and_rejects_oversize(kdt, oracle_mod):
    import torch
    # automatic SIMT splits whose partials exceed the fixed scratch: the library lowers the
    # split count until they fit, and the result still matches
    c, pl = _auto_simt_plan_over_limit(kdt)
    assert c is not None, "no fp32 shape with an automatic split plan above 64 MiB"
    assert pl["impl"] == "simt_small" and pl["num_splits"] > 1
    got, ref = _both(kdt, c, impl="simt_small")
    _check(c, got, ref, oracle_mod)
    # the bf16 tensor path's automatic plan fits as it is
    t = wl.make_case("noalloc_c", B=2, T=64, H=64, prefix=2000, dtype="bf16", tree="geometric", seed=43)
    got, ref = _both(kdt, t, impl="auto")
    _check(t, got, ref, oracle_mod)
    # an explicit split count whose partials exceed the fixed scratch is refused before any launch
    c = t
    d = G.to_device(c)
    out = torch.empty((c.B, c.T, c.H, 512), device="cuda")
    a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                      max_kv_len=c.max_kv_len, scale=c.scale, out=out, impl="simt_small", num_splits=16)
    assert kdt.workspace_size(a) > (64 << 20)
    st = kdt.lib().kdt_verify_attn_noalloc(ctypes.byref(a), None)
    assert st == kdt.kdt.KDT_ERR_WORKSPACE
