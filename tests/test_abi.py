"""CPU checks of the C ABI: the library loads, exports every function include/kdt.h
declares, the ctypes struct matches the C layout, and host-side argument checks
reject bad calls before any launch (none of these calls touch a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def kdt():
    from speculative_decoding_tree_absorb_gb300 import build_lib
    build_lib.build()
    import speculative_decoding_tree_absorb_gb300 as k
    return k


def _declared_functions():
    src = "\n".join(open(h).read() for h in HEADERS)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    names = set(re.findall(r"\b(kdt_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declarations_are_exported(kdt):
    names = _declared_functions()
    assert len(names) >= 7
    lib = kdt.lib()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in kdt.h but not exported by libkdt.so"
    assert set(kdt.EXPORTS) <= set(names)
    nm = subprocess.run(["nm", "-D", "--defined-only", kdt.kdt.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", nm, flags=re.M), n


def test_struct_layout_matches_header(kdt, tmp_path):
    prog = tmp_path / "layout.c"
    fields = [f[0] for f in kdt.VerifyArgs._fields_]
    body = "\n".join(f'printf("{f} %zu\\n", offsetof(kdt_verify_args, {f}));' for f in fields)
    prog.write_text(f"""
#include <stdio.h>
#include <stddef.h>
#include "kdt.h"
int main(void) {{
  printf("size %zu\\n", sizeof(kdt_verify_args));
  printf("plan %zu\\n", sizeof(kdt_plan));
  {body}
  return 0;
}}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include", str(prog),
                    "-o", str(exe)], check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    assert int(out["size"]) == ctypes.sizeof(kdt.VerifyArgs)
    assert int(out["plan"]) == ctypes.sizeof(kdt.kdt.Plan)
    for f in fields:
        assert int(out[f]) == getattr(kdt.VerifyArgs, f).offset, f


def _args(kdt, **kw):
    a = kdt.VerifyArgs()
    a.B, a.T, a.H, a.D_c, a.D_r, a.dtype = 2, 9, 8, 512, 64, 0
    # fake, 256-aligned non-null addresses: only host-side checks run in these tests
    a.q_nope, a.q_pe, a.c_kv, a.k_pe = 0x10000, 0x20000, 0x30000, 0x40000
    a.kv_row_stride, a.prefix_len, a.max_kv_len = 46, 0x50000, 46
    a.parent, a.vis = 0x60000, None
    a.scale, a.out, a.lse, a.err, a.impl, a.num_splits = 0.07, 0x70000, 0x80000, None, 1, 2
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _status(kdt, a):
    return kdt.lib().kdt_verify_attn(ctypes.byref(a), None, 0, None)


def test_host_checks_reject_bad_arguments(kdt):
    K = kdt.kdt
    assert _status(kdt, _args(kdt, D_c=256)) == K.KDT_ERR_UNSUPPORTED
    assert _status(kdt, _args(kdt, D_r=32)) == K.KDT_ERR_UNSUPPORTED
    assert _status(kdt, _args(kdt, dtype=7)) == K.KDT_ERR_UNSUPPORTED
    assert _status(kdt, _args(kdt, impl=9)) == K.KDT_ERR_UNSUPPORTED
    assert _status(kdt, _args(kdt, q_nope=None)) == K.KDT_ERR_NULL_ARG
    assert _status(kdt, _args(kdt, out=None)) == K.KDT_ERR_NULL_ARG
    assert _status(kdt, _args(kdt, parent=None)) == K.KDT_ERR_NULL_ARG           # neither mask input
    assert _status(kdt, _args(kdt, vis=0x90000)) == K.KDT_ERR_NULL_ARG           # both mask inputs
    assert _status(kdt, _args(kdt, T=0)) == K.KDT_ERR_BAD_SHAPE
    assert _status(kdt, _args(kdt, H=0)) == K.KDT_ERR_BAD_SHAPE
    assert _status(kdt, _args(kdt, B=-1)) == K.KDT_ERR_BAD_SHAPE
    assert _status(kdt, _args(kdt, max_kv_len=47)) == K.KDT_ERR_BAD_SHAPE        # beyond the row stride
    assert _status(kdt, _args(kdt, max_kv_len=8)) == K.KDT_ERR_BAD_SHAPE         # below T
    assert _status(kdt, _args(kdt, c_kv=0x30004)) == K.KDT_ERR_BAD_SHAPE         # misaligned
    assert _status(kdt, _args(kdt, num_splits=-1)) == K.KDT_ERR_BAD_SHAPE
    assert _status(kdt, _args(kdt, scale=float("nan"))) == K.KDT_ERR_BAD_SHAPE
    # a valid call without the workspace it needs is refused before launching
    assert _status(kdt, _args(kdt)) == K.KDT_ERR_WORKSPACE
    assert _status(kdt, _args(kdt, B=0)) == K.KDT_OK                             # nothing to do
    lib = kdt.lib()
    assert lib.kdt_build_visibility(None, 2, 0, None, None, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_build_visibility(None, 2, 5, None, None, None) == K.KDT_ERR_NULL_ARG
    assert lib.kdt_merge_attn_states(None, None, None, None, 4, 6, None, None, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_merge_attn_states(None, None, None, None, 4, 512, None, None, None) == K.KDT_ERR_NULL_ARG
    # the w_vc up-projection's host checks (fake device addresses, never dereferenced)
    vc = lib.kdt_vc_up_proj
    assert vc(0x10000, 0x20000, K.KDT_BF16, -1, 4, 512, 128, 0x30000, None, None) == K.KDT_ERR_BAD_SHAPE
    assert vc(0x10000, 0x20000, K.KDT_BF16, 8, 0, 512, 128, 0x30000, None, None) == K.KDT_ERR_BAD_SHAPE
    assert vc(0x10000, 0x20000, K.KDT_BF16, 8, 4, 256, 128, 0x30000, None, None) == K.KDT_ERR_UNSUPPORTED
    assert vc(0x10000, 0x20000, K.KDT_BF16, 8, 4, 512, 100, 0x30000, None, None) == K.KDT_ERR_UNSUPPORTED
    assert vc(0x10000, 0x20000, K.KDT_F32, 8, 4, 512, 128, 0x30000, None, None) == K.KDT_ERR_UNSUPPORTED
    assert vc(None, 0x20000, K.KDT_BF16, 8, 4, 512, 128, 0x30000, None, None) == K.KDT_ERR_NULL_ARG
    assert vc(0x10004, 0x20000, K.KDT_BF16, 8, 4, 512, 128, 0x30000, None, None) == K.KDT_ERR_BAD_SHAPE
    assert vc(None, None, K.KDT_BF16, 0, 4, 512, 128, None, None, None) == K.KDT_OK     # nothing to do
    assert kdt.status_str(K.KDT_ERR_WORKSPACE) == "workspace missing or too small"
    assert kdt.status_str(K.KDT_ERR_NOT_DEVICE).startswith("tensor not in device memory")
    assert lib.kdt_version() >= 100


def test_host_entry_checks(kdt):
    """kdt_verify_attn_host refuses bad arguments, chunk counts, streams and buffers before
    any CUDA call (the stream handles below are never used)."""
    K = kdt.kdt
    lib = kdt.lib()

    def host(a, n=0, buf=None, nbytes=0, streams=(1, 2, 3)):
        return lib.kdt_verify_attn_host(ctypes.byref(a), n, buf, nbytes, *(ctypes.c_void_p(x) for x in streams))

    def size(a, n=0):
        return lib.kdt_verify_attn_host_buffer_size(ctypes.byref(a), n)

    a = _args(kdt)                                     # B = 2, fp32, parent given: two chunks by default
    need = size(a)
    per_seq = (9 * 8 * 576 * 4 + 46 * 576 * 4 + 4 + 9 * 4) + (9 * 8 * 512 * 4 + 9 * 8 * 4)
    assert need >= 2 * per_seq + kdt.workspace_size(_args(kdt, B=1))
    assert size(a, 1) >= 2 * per_seq and size(a, 2) == need
    assert host(a) == K.KDT_ERR_WORKSPACE                                   # no buffer
    assert host(a, buf=0x100000, nbytes=need - 1) == K.KDT_ERR_WORKSPACE   # short
    assert host(a, buf=0x100010, nbytes=need) == K.KDT_ERR_WORKSPACE       # not 256-byte aligned
    assert host(a, n=3) == K.KDT_ERR_BAD_SHAPE and size(a, 3) == 0          # does not divide B
    assert host(a, n=-1) == K.KDT_ERR_BAD_SHAPE
    assert host(_args(kdt, q_nope_row_stride=576)) == K.KDT_ERR_BAD_SHAPE   # host rows are contiguous
    for streams in ((1, 1, 3), (1, 2, 1), (1, 2, 2)):
        assert host(a, buf=0x100000, nbytes=need, streams=streams) == K.KDT_ERR_BAD_SHAPE
    assert host(_args(kdt, out=None)) == K.KDT_ERR_NULL_ARG
    assert host(_args(kdt, D_c=256)) == K.KDT_ERR_UNSUPPORTED and size(_args(kdt, D_c=256)) == 0
    assert host(_args(kdt, B=0)) == K.KDT_OK and size(_args(kdt, B=0)) == 0
    # one sequence a chunk needs room for every chunk's tensors
    b = _args(kdt, B=4)
    assert size(b, 4) >= 4 * per_seq and size(b, 0) == size(b, 4)


def test_plan_and_workspace_are_host_only(kdt):
    a = _args(kdt, num_splits=3)
    p = kdt.plan(a)
    # the 64-row SIMT tile: 3 CTAs share the 4 (row tile, key block) pairs (2 sequences of
    # 72 rows, one 128-key block each) and leave piece states for a merge
    assert p["impl"] == "simt" and p["num_splits"] == 3
    assert p["num_launches"] == 3                                  # visibility + attention + merge
    assert kdt.workspace_size(a) == p["workspace_bytes"] >= 2 * 9 * 4 + 2 * 3 * 64 * 513 * 4
    assert kdt.plan(_args(kdt, num_splits=9))["num_splits"] == 4   # never more CTAs than pairs
    # the small-shape path: 46 keys fit one 64-key block, so one pass a CTA with the
    # visibility built in the kernel: one launch, no workspace; its 2 x 72 rows fit one
    # wave at one row a CTA (one fp32 CTA an SM, at least 148 SMs)
    s = kdt.plan(_args(kdt, impl=3, num_splits=3))
    assert s["impl"] == "simt_small" and s["num_splits"] == 1 and s["num_launches"] == 1
    assert s["workspace_bytes"] == 0 and s["ctas"] == 2 * 72
    # more rows than SMs: 2, then 4 rows a CTA (the grid of the fewest rows that fits one wave)
    assert kdt.plan(_args(kdt, impl=3, H=16))["ctas"] == 2 * 72
    assert kdt.plan(_args(kdt, impl=3, H=64))["ctas"] == 2 * 144
    # longer caches take the 16-row tile, one 64-key block per split
    s = kdt.plan(_args(kdt, impl=3, kv_row_stride=200, max_kv_len=200, num_splits=0))
    assert s["impl"] == "simt_small" and s["num_splits"] == 4 and s["num_launches"] == 3
    b = _args(kdt, kv_row_stride=4096 + 32, max_kv_len=4096 + 32, T=32, H=64, B=1, num_splits=8, vis=0x90000,
              parent=None)
    p = kdt.plan(b)
    # the 64-row SIMT tile shares its (row tile, key block) pairs over the asked 8 CTAs,
    # each leaving at most two piece states of 64 rows for the merge
    assert p["num_splits"] == 8 and p["num_launches"] == 2        # attention + merge
    assert p["workspace_bytes"] >= 2 * 8 * 64 * 512 * 4 + 2 * 8 * 64 * 4
    assert kdt.workspace_size(_args(kdt, D_c=3)) == 0
    # bf16 inputs plan onto the tensor-core kernel: one 4-CTA cluster per resident slot (at
    # most 48), sharing all units' key blocks; units cut by the split leave piece states in
    # the workspace
    c = _args(kdt, dtype=1, impl=0, B=8, T=64, H=64, kv_row_stride=8256, max_kv_len=8256, num_splits=1)
    p = kdt.plan(c)
    assert p["impl"] == "tcgen05" and p["ctas"] % 4 == 0 and 4 <= p["ctas"] <= 4 * 48 and p["num_splits"] == 1
    clusters = p["ctas"] // 4
    if clusters > 1:
        assert p["workspace_bytes"] >= 2 * clusters * 256 * (512 + 1) * 4 and p["num_launches"] == 3
    assert _status(kdt, _args(kdt, dtype=0, impl=2)) == kdt.kdt.KDT_ERR_UNSUPPORTED   # fp32 on tensor cores


def test_tree_op_host_checks(kdt):
    lib = kdt.lib()
    K = kdt.kdt
    assert lib.kdt_tree_accept(None, None, None, -1, 4, None, None, None, None, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_tree_accept(None, None, None, 2, 0, None, None, None, None, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_tree_accept(None, None, None, 2, 5, None, None, None, None, None) == K.KDT_ERR_NULL_ARG
    assert lib.kdt_kv_compact(None, None, K.KDT_BF16, 512, 64, 2, 5, 3, None, None, None, 1, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_kv_compact(None, None, K.KDT_BF16, 500, 64, 2, 5, 100, None, None, None, 1, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_kv_compact(None, None, 7, 512, 64, 2, 5, 100, None, None, None, 1, None) == K.KDT_ERR_UNSUPPORTED
    assert lib.kdt_kv_compact(None, None, K.KDT_BF16, 512, 64, 2, 5, 100, None, None, None, 1, None) == K.KDT_ERR_NULL_ARG
    a = K.RopeArgs()
    a.B, a.T, a.H, a.D_r, a.dtype, a.base = 2, 4, 8, 63, K.KDT_BF16, 10000.0
    assert lib.kdt_rope_neox(ctypes.byref(a), None) == K.KDT_ERR_BAD_SHAPE
    a.D_r = 64
    assert lib.kdt_rope_neox(ctypes.byref(a), None) == K.KDT_ERR_NULL_ARG
    a.base = -1.0
    assert lib.kdt_rope_neox(ctypes.byref(a), None) == K.KDT_ERR_BAD_SHAPE


def test_tree_build_host_checks(kdt):
    lib = kdt.lib()
    K = kdt.kdt
    assert lib.kdt_tree_build(None, None, 1, 0, 4, 3, None, None, None, None, None, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_tree_build(None, None, 1, 4, 33, 3, None, None, None, None, None, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_tree_build(None, None, 1, 2, 2, 7, None, None, None, None, None, None) == K.KDT_ERR_BAD_SHAPE
    assert lib.kdt_tree_build(None, None, 1, 2, 2, 6, None, None, None, None, None, None) == K.KDT_ERR_NULL_ARG
    assert lib.kdt_tree_build(None, None, 1, 64, 32, 4096, None, None, None, None, None, None) == K.KDT_ERR_BAD_SHAPE
