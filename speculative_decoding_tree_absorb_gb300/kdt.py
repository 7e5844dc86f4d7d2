"""Thin Python binding of libkdt.so (ctypes). Argument marshalling only.

Every computation runs in the library's CUDA kernels; this module passes device
pointers (``tensor.data_ptr()``) and the current CUDA stream, and allocates
output and workspace tensors with torch when the caller does not pass them.
There is no CPU fallback: if libkdt.so is missing, importing the library raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkdt.so")

(KDT_OK, KDT_ERR_NULL_ARG, KDT_ERR_BAD_SHAPE, KDT_ERR_UNSUPPORTED, KDT_ERR_WORKSPACE, KDT_ERR_CUDA,
 KDT_ERR_NOT_DEVICE) = range(7)
KDT_F32, KDT_BF16 = 0, 1
IMPLS = {"auto": 0, "simt": 1, "tcgen05": 2, "simt_small": 3}
IMPL_NAMES = {v: k for k, v in IMPLS.items()}
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)

# Names the header declares (checked by the CPU test suite against include/kdt.h).
EXPORTS = ("kdt_status_str", "kdt_version", "kdt_build_visibility", "kdt_verify_attn",
           "kdt_verify_attn_workspace_size", "kdt_verify_attn_plan", "kdt_merge_attn_states",
           "kdt_verify_attn_noalloc", "kdt_rope_neox", "kdt_tree_accept", "kdt_kv_compact", "kdt_tree_build",
           "kdt_verify_attn_host", "kdt_verify_attn_host_buffer_size", "kdt_vc_up_proj",
           "kdt_test_verify_attn_wait_expiry")


class KdtError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


class VerifyArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("D_c", ctypes.c_int), ("D_r", ctypes.c_int), ("dtype", ctypes.c_int),
        ("q_nope", ctypes.c_void_p), ("q_pe", ctypes.c_void_p),
        ("c_kv", ctypes.c_void_p), ("k_pe", ctypes.c_void_p),
        ("kv_row_stride", ctypes.c_int64),
        ("prefix_len", ctypes.c_void_p),
        ("max_kv_len", ctypes.c_int),
        ("parent", ctypes.c_void_p), ("vis", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("err", ctypes.c_void_p),
        ("impl", ctypes.c_int), ("num_splits", ctypes.c_int),
        ("q_nope_row_stride", ctypes.c_int64), ("q_pe_row_stride", ctypes.c_int64),
    ]


class RopeArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("D_r", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("q", ctypes.c_void_p), ("q_row_stride", ctypes.c_int64),
        ("k_pe", ctypes.c_void_p), ("kv_row_stride", ctypes.c_int64),
        ("prefix_len", ctypes.c_void_p), ("pos", ctypes.c_void_p),
        ("base", ctypes.c_double),
    ]


class Plan(ctypes.Structure):
    _fields_ = [("impl", ctypes.c_int), ("num_splits", ctypes.c_int), ("num_launches", ctypes.c_int),
                ("ctas", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def lib():
    """The loaded libkdt.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkdt.so not found at {LIB_PATH}: build it with "
                              "`python -m speculative_decoding_tree_absorb_gb300.build_lib` "
                              "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp = ctypes.c_void_p
        L.kdt_status_str.argtypes = [ctypes.c_int]
        L.kdt_status_str.restype = ctypes.c_char_p
        L.kdt_version.argtypes = []
        L.kdt_version.restype = ctypes.c_int
        L.kdt_build_visibility.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        L.kdt_build_visibility.restype = ctypes.c_int
        L.kdt_verify_attn.argtypes = [ctypes.POINTER(VerifyArgs), vp, ctypes.c_size_t, vp]
        L.kdt_verify_attn.restype = ctypes.c_int
        L.kdt_verify_attn_workspace_size.argtypes = [ctypes.POINTER(VerifyArgs)]
        L.kdt_verify_attn_workspace_size.restype = ctypes.c_size_t
        L.kdt_verify_attn_plan.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.POINTER(Plan)]
        L.kdt_verify_attn_plan.restype = ctypes.c_int
        L.kdt_merge_attn_states.argtypes = [vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int, vp, vp, vp]
        L.kdt_merge_attn_states.restype = ctypes.c_int
        L.kdt_verify_attn_host.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.c_int, vp, ctypes.c_size_t, vp, vp, vp]
        L.kdt_verify_attn_host.restype = ctypes.c_int
        L.kdt_verify_attn_host_buffer_size.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.c_int]
        L.kdt_verify_attn_host_buffer_size.restype = ctypes.c_size_t
        L.kdt_vc_up_proj.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     vp, vp, vp]
        L.kdt_vc_up_proj.restype = ctypes.c_int
        L.kdt_test_verify_attn_wait_expiry.argtypes = [ctypes.POINTER(VerifyArgs), vp, ctypes.c_size_t,
                                                       ctypes.c_uint32, vp]
        L.kdt_test_verify_attn_wait_expiry.restype = ctypes.c_int
        L.kdt_verify_attn_noalloc.argtypes = [ctypes.POINTER(VerifyArgs), vp]
        L.kdt_verify_attn_noalloc.restype = ctypes.c_int
        L.kdt_rope_neox.argtypes = [ctypes.POINTER(RopeArgs), vp]
        L.kdt_rope_neox.restype = ctypes.c_int
        L.kdt_tree_accept.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp]
        L.kdt_tree_accept.restype = ctypes.c_int
        L.kdt_kv_compact.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int64, vp, vp, vp, ctypes.c_int, vp]
        L.kdt_kv_compact.restype = ctypes.c_int
        L.kdt_tree_build.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp,
                                     vp, vp]
        L.kdt_tree_build.restype = ctypes.c_int
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().kdt_status_str(int(status)).decode()


def _check(status: int, where: str):
    if status != KDT_OK:
        raise KdtError(status, where)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return KDT_F32
    if t.dtype == torch.bfloat16:
        return KDT_BF16
    raise TypeError(f"inputs must be float32 or bfloat16, got {t.dtype}")


def make_args(q_nope, q_pe, c_kv, k_pe, prefix_len, *, parent=None, vis=None, max_kv_len=None,
              scale=DEFAULT_SCALE, out=None, lse=None, err=None, impl="auto", num_splits=0) -> VerifyArgs:
    """Fill the C argument struct from tensors (no checks beyond what the library does)."""
    B, T, H = q_nope.shape[0], q_nope.shape[1], q_nope.shape[2]
    L = c_kv.shape[1]
    a = VerifyArgs()
    a.B, a.T, a.H = B, T, H
    a.D_c, a.D_r = q_nope.shape[3], q_pe.shape[3]
    a.dtype = _dtype_code(q_nope)
    a.q_nope, a.q_pe, a.c_kv, a.k_pe = (t.data_ptr() for t in (q_nope, q_pe, c_kv, k_pe))
    a.kv_row_stride = L
    a.prefix_len = prefix_len.data_ptr()
    a.max_kv_len = int(L if max_kv_len is None else max_kv_len)
    a.parent = None if parent is None else parent.data_ptr()
    a.vis = None if vis is None else vis.data_ptr()
    a.scale = float(scale)
    a.out = None if out is None else out.data_ptr()
    a.lse = None if lse is None else lse.data_ptr()
    a.err = None if err is None else err.data_ptr()
    a.impl = IMPLS[impl] if isinstance(impl, str) else int(impl)
    a.num_splits = int(num_splits)
    a.q_nope_row_stride = _row_stride(q_nope)
    a.q_pe_row_stride = _row_stride(q_pe)
    return a


def _row_stride(q):
    """0 for a contiguous [B,T,H,d] tensor; else the element stride between (b,i,h) rows
    of a view with a contiguous last dim and equally spaced rows (e.g. a slice of a
    combined [B,T,H,576] query buffer)."""
    if q.is_contiguous():
        return 0
    if q.stride(3) != 1 or q.stride(2) * q.shape[2] != q.stride(1) or q.stride(1) * q.shape[1] != q.stride(0):
        raise ValueError("query views must have a contiguous last dim and equally spaced (b,i,h) rows")
    return int(q.stride(2))


def plan(args: VerifyArgs) -> dict:
    p = Plan()
    _check(lib().kdt_verify_attn_plan(ctypes.byref(args), ctypes.byref(p)), "kdt_verify_attn_plan")
    return dict(impl=IMPL_NAMES.get(p.impl, p.impl), num_splits=p.num_splits, num_launches=p.num_launches,
                ctas=p.ctas, workspace_bytes=int(p.workspace_bytes))


def workspace_size(args: VerifyArgs) -> int:
    return int(lib().kdt_verify_attn_workspace_size(ctypes.byref(args)))


def build_visibility(parent, err=None, stream=None):
    """parent int32 [B,T] (cuda) -> packed bits uint32-as-int32 tensor [B,T,ceil(T/32)]."""
    import torch
    B, T = parent.shape
    vis = torch.empty((B, T, (T + 31) // 32), dtype=torch.int32, device=parent.device)
    _check(lib().kdt_build_visibility(_ptr(parent), B, T, _ptr(vis), _ptr(err), _stream_ptr(stream)),
           "kdt_build_visibility")
    return vis


def verify_attn(q_nope, q_pe, c_kv, k_pe, prefix_len, *, parent=None, vis=None, max_kv_len=None,
                scale=DEFAULT_SCALE, out=None, lse=None, err=None, impl="auto", num_splits=0,
                workspace=None, stream=None, want_lse=True):
    """Tree-verify MLA-absorb attention. Returns (out [B,T,H,512] fp32, lse [B,T,H] fp32 or None).

    ``max_kv_len`` defaults to the cache row stride (c_kv.shape[1]), a valid host
    bound that needs no device->host read of prefix_len.
    """
    import torch
    B, T, H = q_nope.shape[:3]
    dev = q_nope.device
    if out is None:
        out = torch.empty((B, T, H, q_nope.shape[3]), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    a = make_args(q_nope, q_pe, c_kv, k_pe, prefix_len, parent=parent, vis=vis, max_kv_len=max_kv_len,
                  scale=scale, out=out, lse=lse, err=err, impl=impl, num_splits=num_splits)
    need = workspace_size(a)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kdt_verify_attn(ctypes.byref(a), _ptr(workspace), ws_bytes, _stream_ptr(stream)),
           "kdt_verify_attn")
    return out, lse


def host_buffer_size(args: VerifyArgs, n_chunks=0) -> int:
    return int(lib().kdt_verify_attn_host_buffer_size(ctypes.byref(args), int(n_chunks)))


def verify_attn_host(q_nope, q_pe, c_kv, k_pe, prefix_len, *, parent=None, vis=None, max_kv_len=None,
                     scale=DEFAULT_SCALE, out=None, lse=None, err=None, impl="auto", num_splits=0, n_chunks=0,
                     dev_buf=None, streams=None, want_lse=True, device=None):
    """kdt_verify_attn_host: host (CPU, ideally pinned) tensors in, host out and lse back.

    ``streams`` = (compute, copy in, copy out) torch streams (default: the current
    stream and two new ones); ``dev_buf`` a device uint8 tensor of at least
    host_buffer_size() bytes (allocated here if None). The result is complete once
    the compute stream is synchronised. ``err`` is a device int32 word."""
    import torch
    B, T, H = q_nope.shape[:3]
    dev = torch.device("cuda") if device is None else torch.device(device)
    if out is None:
        out = torch.empty((B, T, H, q_nope.shape[3]), dtype=torch.float32, pin_memory=True)
    if lse is None and want_lse:
        lse = torch.empty((B, T, H), dtype=torch.float32, pin_memory=True)
    a = make_args(q_nope, q_pe, c_kv, k_pe, prefix_len, parent=parent, vis=vis, max_kv_len=max_kv_len,
                  scale=scale, out=out, lse=lse, err=err, impl=impl, num_splits=num_splits)
    need = host_buffer_size(a, n_chunks)
    if dev_buf is None and need > 0:
        dev_buf = torch.empty(need, dtype=torch.uint8, device=dev)
    nbytes = 0 if dev_buf is None else dev_buf.numel() * dev_buf.element_size()
    if streams is None:
        streams = (torch.cuda.current_stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    s, s_in, s_out = (ctypes.c_void_p(x.cuda_stream) for x in streams)
    _check(lib().kdt_verify_attn_host(ctypes.byref(a), int(n_chunks), _ptr(dev_buf), nbytes, s, s_in, s_out),
           "kdt_verify_attn_host")
    return out, lse


def merge_attn_states(o_a, lse_a, o_b, lse_b, out=None, lse=None, stream=None):
    """Log-sum-exp merge of two attention states over disjoint key sets."""
    import torch
    D = o_a.shape[-1]
    rows = lse_a.numel()
    if out is None:
        out = torch.empty_like(o_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    _check(lib().kdt_merge_attn_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, D, _ptr(out),
                                       _ptr(lse), _stream_ptr(stream)), "kdt_merge_attn_states")
    return out, lse


def vc_up_proj(o, w_vc, out=None, err=None, stream=None):
    """Per-head value up-projection (kdt_vc_up_proj): o fp32 [..., H, 512] (e.g. the
    verify output [B,T,H,512]), w_vc bf16 [H, 512, D_v] -> fp32 [..., H, D_v]."""
    import torch
    H, D_c = o.shape[-2], o.shape[-1]
    D_v = w_vc.shape[-1]
    if tuple(w_vc.shape[:2]) != (H, D_c):
        raise ValueError("w_vc must be [H, D_c, D_v] matching o [..., H, D_c]")
    R = o.numel() // (H * D_c) if o.numel() else 0
    if out is None:
        out = torch.empty(tuple(o.shape[:-1]) + (D_v,), dtype=torch.float32, device=o.device)
    _check(lib().kdt_vc_up_proj(_ptr(o), _ptr(w_vc), _dtype_code(w_vc), R, H, D_c, D_v, _ptr(out), _ptr(err),
                                _stream_ptr(stream)), "kdt_vc_up_proj")
    return out


def verify_attn_noalloc(q_nope, q_pe, c_kv, k_pe, prefix_len, *, out, lse=None, parent=None, vis=None,
                        max_kv_len=None, scale=DEFAULT_SCALE, err=None, impl="auto", num_splits=0, stream=None):
    """kdt_verify_attn_noalloc: the same attention with the library's fixed scratch array.

    For callers that must not allocate device memory at call time: the caller passes
    every input and output (``out`` is required); the library neither allocates nor
    asks for a workspace. Calls on one device share the scratch array, so calls
    that overlap on the GPU race; see include/kdt.h.
    """
    a = make_args(q_nope, q_pe, c_kv, k_pe, prefix_len, parent=parent, vis=vis, max_kv_len=max_kv_len,
                  scale=scale, out=out, lse=lse, err=err, impl=impl, num_splits=num_splits)
    _check(lib().kdt_verify_attn_noalloc(ctypes.byref(a), _stream_ptr(stream)), "kdt_verify_attn_noalloc")
    return out, lse


def rope_neox(pos, *, q=None, k_pe=None, prefix_len=None, base=10000.0, stream=None):
    """NeoX rotary embedding in place (kdt_rope_neox).

    ``q``: a [B,T,H,d] view whose last dim is contiguous -- e.g. the rope slice
    ``q_comb[..., 512:]`` of a combined [B,T,H,576] query buffer (its row stride is
    taken from the view). ``k_pe``: the [B,L,d] key cache; rows prefix_len[b] + i are
    rotated. ``pos`` int32 [B,T]. Returns nothing: the tensors are updated in place.
    """
    a = RopeArgs()
    a.B, a.T = pos.shape
    ref = q if q is not None else k_pe
    a.dtype = _dtype_code(ref)
    if q is not None:
        if q.stride(3) != 1 or q.stride(2) * q.shape[2] != q.stride(1) or q.stride(1) * q.shape[1] != q.stride(0):
            raise ValueError("q must be a [B,T,H,d] view with equally spaced (b,i,h) rows and a contiguous last dim")
        a.H, a.D_r = q.shape[2], q.shape[3]
        a.q, a.q_row_stride = q.data_ptr(), q.stride(2)
    else:
        a.H, a.D_r = 1, k_pe.shape[2]
    if k_pe is not None:
        a.k_pe, a.kv_row_stride = k_pe.data_ptr(), k_pe.shape[1]
        a.prefix_len = None if prefix_len is None else prefix_len.data_ptr()
    a.pos = pos.data_ptr()
    a.base = float(base)
    _check(lib().kdt_rope_neox(ctypes.byref(a), _stream_ptr(stream)), "kdt_rope_neox")


def tree_accept(parent, tok, target, err=None, stream=None):
    """Greedy accept walk (kdt_tree_accept). Returns (acc_nodes [B,T], n_acc [B], bonus [B]) int32."""
    import torch
    B, T = parent.shape
    dev = parent.device
    acc = torch.empty((B, T), dtype=torch.int32, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    bonus = torch.empty(B, dtype=torch.int32, device=dev)
    _check(lib().kdt_tree_accept(_ptr(parent), _ptr(tok), _ptr(target), B, T, _ptr(acc), _ptr(n), _ptr(bonus),
                                 _ptr(err), _stream_ptr(stream)), "kdt_tree_accept")
    return acc, n, bonus


def kv_compact(c_kv, k_pe, prefix_len, acc_nodes, n_acc, update_prefix=True, stream=None):
    """Move the accepted path's cache rows to prefix_len + k, in place (kdt_kv_compact)."""
    B, T = acc_nodes.shape
    _check(lib().kdt_kv_compact(_ptr(c_kv), _ptr(k_pe), _dtype_code(c_kv), c_kv.shape[2], k_pe.shape[2], B, T,
                                c_kv.shape[1], _ptr(prefix_len), _ptr(acc_nodes), _ptr(n_acc),
                                1 if update_prefix else 0, _stream_ptr(stream)), "kdt_kv_compact")


def tree_build(cand_tok, cand_lp, N, root_tok=None, stream=None):
    """Best-first draft tree (kdt_tree_build). cand_tok int32 / cand_lp float32 [B,D,K].
    Returns (parent, tok, depth) int32 [B,N+1] and score float32 [B,N+1]."""
    import torch
    B, D, K = cand_lp.shape
    dev = cand_lp.device
    parent = torch.empty((B, N + 1), dtype=torch.int32, device=dev)
    tok = torch.empty_like(parent)
    depth = torch.empty_like(parent)
    score = torch.empty((B, N + 1), dtype=torch.float32, device=dev)
    _check(lib().kdt_tree_build(_ptr(cand_tok), _ptr(cand_lp), B, D, K, int(N), _ptr(root_tok), _ptr(parent),
                                _ptr(tok), _ptr(depth), _ptr(score), _stream_ptr(stream)), "kdt_tree_build")
    return parent, tok, depth, score
