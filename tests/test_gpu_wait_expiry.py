"""The tensor-core kernel's bounded waits, exercised on the GPU without a fault.

Every pipeline wait in the kernel gives up after a time limit, records a negative code
in the caller's error word, and lets the kernel leave cleanly (in-flight copies and MMAs
drained, tensor memory freed). A test hook (kdt_test_verify_attn_wait_expiry, declared in
include/kdt_testing.h) withholds the first work item's Q-ready arrivals -- a barrier that
nothing else completes -- and cuts the limit to a few milliseconds. The call must end in
well under a second with a negative error code, the CUDA context must stay usable, and
the next normal call on the same context must match the oracle (a kernel that left its
tensor memory allocated would block the next one instead)."""
import ctypes
import time

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


@pytest.mark.parametrize("clusters", [1, 4])
def test_expired_wait_is_reported_and_the_context_stays_usable(kdt, oracle_mod, clusters):
    import torch
    case = wl.make_case("expiry", B=2, T=16, H=64, prefix=(300, 517), dtype="bf16", tree="geometric", seed=3)
    d = G.to_device(case)
    out = torch.full((case.B, case.T, case.H, 512), float("nan"), device="cuda")
    lse = torch.empty((case.B, case.T, case.H), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                      max_kv_len=case.max_kv_len, scale=case.scale, out=out, lse=lse, err=err, impl="tcgen05",
                      num_splits=clusters)
    ws = torch.empty(max(1, kdt.workspace_size(a)), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = kdt.lib().kdt_test_verify_attn_wait_expiry(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                                     2000, None)
    torch.cuda.synchronize()                      # raises if the context were lost
    elapsed = time.perf_counter() - t0
    assert st == kdt.kdt.KDT_OK
    code = int(err.item())
    assert code < 0, f"expected a negative wait-expiry code, got {code}"
    assert elapsed < 2.0, f"the failed call took {elapsed:.3f} s"
    # the same context, the same inputs, a normal call: complete and oracle-exact
    ref_out, ref_lse = oracle_mod.verify_attn(case)
    for _ in range(2):
        got_out, got_lse, e = G.run(case, impl="tcgen05", num_splits=clusters, dev_tensors=d)
        assert e == 0
        H.assert_close(got_out, ref_out, *H.TOL["bf16"], what="after expiry out")
        H.assert_close(got_lse, ref_lse, *H.TOL["bf16"], what="after expiry lse")


def test_hook_refuses_the_simt_kernel(kdt):
    import torch
    case = wl.make_case("expiry32", B=1, T=4, H=8, prefix=40, dtype="f32", tree="geometric", seed=3)
    d = G.to_device(case)
    out = torch.empty((case.B, case.T, case.H, 512), device="cuda")
    a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                      max_kv_len=case.max_kv_len, out=out)
    ws = torch.empty(max(1, kdt.workspace_size(a)), dtype=torch.uint8, device="cuda")
    st = kdt.lib().kdt_test_verify_attn_wait_expiry(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                                     2000, None)
    assert st == kdt.kdt.KDT_ERR_UNSUPPORTED
