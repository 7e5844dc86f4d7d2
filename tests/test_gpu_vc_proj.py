"""GPU parity of the per-head w_vc up-projection (kdt_vc_up_proj) against the oracle,
through the C ABI. The kernel is fp32-accurate (the fp32 latent split into two bf16
parts, bf16 weights exact), so it is held to the fp32 bound |gpu - oracle| <=
1e-4 + 1e-4 |oracle| on every element."""
import numpy as np
import pytest

import workloads as wl
from oracle import tree_ops as ot
from tests import gpu_util as G
from tests import helpers as H

pytestmark = pytest.mark.gpu

TOL = H.TOL["f32"]


@pytest.fixture(scope="module")
def kdt():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_absorb_gb300 import build_lib
    build_lib.build()
    import speculative_decoding_tree_absorb_gb300 as k
    return k


def _inputs(seed, R, Hh, D_v, sigma_o=1.0):
    o = wl.normal(seed, "vc_o", R * Hh * 512, sigma_o).reshape(R, Hh, 512).astype(np.float32)
    w = wl.f64_to_bf16_bits(wl.normal(seed, "vc_w", Hh * 512 * D_v, 1.0 / np.sqrt(512.0))).reshape(Hh, 512, D_v)
    return o, w


def _run(kdt, o, w):
    import torch
    err = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    w_d = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).cuda()
    v = kdt.vc_up_proj(torch.from_numpy(o).cuda(), w_d, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return v.cpu().numpy()


@pytest.mark.parametrize("R,Hh,D_v", [(1, 1, 128), (5, 3, 128), (9, 2, 128), (127, 2, 64), (128, 4, 128),
                                      (129, 3, 128), (300, 5, 64), (512, 8, 128), (999, 3, 128), (1000, 2, 128),
                                      (601, 50, 64)])
def test_vc_up_proj_matches_oracle(kdt, R, Hh, D_v):
    # R % 8 != 0 leaves a short last group in every head; with H*ceil(R/8) groups shared by
    # up to one CTA per SM, shares start and end inside heads and inside 128-row spans
    # ((999, 3): two or three groups a CTA; (601, 50): about 25, cut at head ends)
    o, w = _inputs(R * 7 + Hh, R, Hh, D_v)
    got = _run(kdt, o, w)
    H.assert_close(got, ot.vc_up_proj(o, w), *TOL, what=f"vc R={R} H={Hh} D_v={D_v}")


@pytest.mark.parametrize("name", ["target", "dsv3"])
def test_vc_up_proj_full_size(kdt, name):
    # the verify output shapes of the target (R = 8*64 rows, H = 64) and DSv3 (R = 16*64,
    # H = 128) workloads, D_v = 128: every element against the oracle
    sh = wl.config_shape(name)
    R, Hh = sh["B"] * sh["T"], sh["H"]
    o, w = _inputs(55, R, Hh, 128, sigma_o=0.1)
    got = _run(kdt, o, w)
    H.assert_close(got, ot.vc_up_proj(o, w), *TOL, what=f"vc {name}")


def test_vc_up_proj_of_verify_output(kdt, oracle_mod):
    # the step as it follows verify: the device's verify output, projected on the device,
    # against the oracle's projection of that same output (copied to the host); and the
    # verify output itself against the oracle's
    import torch
    case = wl.make_case("vc_chain", B=2, T=24, H=16, prefix=(700, 333), dtype="bf16", tree="geometric", seed=9)
    d = G.to_device(case)
    out, lse = kdt.verify_attn(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                               max_kv_len=case.max_kv_len, scale=case.scale)
    _, w = _inputs(3, 1, case.H, 128)
    w_d = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).cuda()
    v = kdt.vc_up_proj(out, w_d)
    torch.cuda.synchronize()
    ref_out, _ = oracle_mod.verify_attn(case)
    H.assert_close(out.cpu().numpy(), ref_out, *H.TOL["bf16"], what="verify out")
    H.assert_close(v.cpu().numpy(), ot.vc_up_proj(out.cpu().numpy(), w), *TOL, what="vc of verify out")


def test_vc_up_proj_one_hot_weights_are_exact(kdt):
    # one-hot weights select latent dims: only the split of o into two bf16 parts is
    # involved (hi = bf16(o) is off by at most 2^-8 |o|, and lo = bf16(o - hi) by 2^-8 of
    # that), so the result equals the selected dims to within 2^-16 of their magnitude
    Hh, R = 2, 200
    o = wl.normal(4, "vc_sel", R * Hh * 512).reshape(R, Hh, 512).astype(np.float32)
    sel = np.stack([(np.arange(128) * 5 + 11 * h) % 512 for h in range(Hh)])
    w = np.zeros((Hh, 512, 128))
    for h in range(Hh):
        w[h, sel[h], np.arange(128)] = 1.0
    got = _run(kdt, o, wl.f64_to_bf16_bits(w))
    for h in range(Hh):
        want = o[:, h, sel[h]].astype(np.float64)
        assert np.all(np.abs(got[:, h] - want) <= 2.0 ** -16 * np.abs(want) + 1e-30)


def test_vc_up_proj_refuses_host_memory_and_bad_sizes(kdt):
    import ctypes
    import torch
    K = kdt.kdt
    o, w = _inputs(1, 16, 2, 128)
    w_d = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).cuda()
    o_d = torch.from_numpy(o).cuda()
    v = torch.full((16, 2, 128), float("nan"), device="cuda")
    lib = kdt.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())      # noqa: E731
    o_h = torch.from_numpy(o).pin_memory()
    assert lib.kdt_vc_up_proj(p(o_h), p(w_d), K.KDT_BF16, 16, 2, 512, 128, p(v), None, None) == K.KDT_ERR_NOT_DEVICE
    assert lib.kdt_vc_up_proj(p(o_d), p(w_d), K.KDT_BF16, 16, 2, 512, 96, p(v), None, None) == K.KDT_ERR_UNSUPPORTED
    assert lib.kdt_vc_up_proj(p(o_d), p(w_d), K.KDT_F32, 16, 2, 512, 128, p(v), None, None) == K.KDT_ERR_UNSUPPORTED
    assert lib.kdt_vc_up_proj(p(o_d), p(w_d), K.KDT_BF16, 0, 2, 512, 128, p(v), None, None) == K.KDT_OK
    torch.cuda.synchronize()
    assert torch.isnan(v).all()                           # nothing ran
