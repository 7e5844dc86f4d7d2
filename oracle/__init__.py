"""CPU oracle for tree-verify MLA-absorb attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library's CUDA path never calls it and
shares no code with it; this wrapper only marshals numpy arrays into the plain C
double-precision implementation in ``kdt_oracle.c`` (built with gcc on first use).

Every function here computes the plain definition stated in ``kdt_oracle.c``.
Parity status per function (how each is pinned is in ``tests/test_oracle.py``):
  build_visibility   -- pinned (exhaustive brute force, T <= 6; chain/star shapes)
  verify_attn*       -- pinned (library softmax on causal and dense masks, path
                        sets on all trees T <= 5, single-key exactness, closed forms
                        for q = 0 from tests/golden, permutation and split invariants)
  attn_weights       -- pinned (sum to 1, exact zeros off the visible set)
  merge_states       -- pinned (split-prefix merge equals the unsplit result)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kdt_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkdt_oracle.so")
_lock = threading.Lock()
_lib = None

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_ll = ctypes.c_longlong
_c_double = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kdt_ref_build_visibility.argtypes = [_c_void_p, _c_int, _c_int, _c_void_p]
            lib.kdt_ref_build_visibility.restype = _c_int
            common = [_c_int, _c_int, _c_int, _c_int, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                      _c_ll, _c_void_p, _c_void_p, _c_void_p, _c_double]
            lib.kdt_ref_verify_attn.argtypes = common + [_c_void_p, _c_void_p, _c_int]
            lib.kdt_ref_verify_attn.restype = _c_int
            lib.kdt_ref_verify_attn_rows.argtypes = common + [_c_void_p, _c_ll, _c_void_p, _c_void_p,
                                                              _c_void_p, _c_void_p, _c_int]
            lib.kdt_ref_verify_attn_rows.restype = _c_int
            lib.kdt_ref_attn_weights.argtypes = common + [_c_ll, _c_void_p]
            lib.kdt_ref_attn_weights.restype = _c_int
            lib.kdt_ref_merge_states.argtypes = [_c_ll, _c_int] + [_c_void_p] * 6
            lib.kdt_ref_merge_states.restype = None
            lib.kdt_ref_num_threads.argtypes = []
            lib.kdt_ref_num_threads.restype = _c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_c_void_p)


def num_threads() -> int:
    return int(_load().kdt_ref_num_threads())


class OracleError(RuntimeError):
    pass


def build_visibility(parent: np.ndarray) -> np.ndarray:
    """parent int32 [B,T] -> packed visibility words uint32 [B,T,ceil(T/32)]."""
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    B, T = parent.shape
    W = (T + 31) // 32
    vis = np.zeros((B, T, W), dtype=np.uint32)
    rc = _load().kdt_ref_build_visibility(_ptr(parent), B, T, _ptr(vis))
    if rc:
        raise OracleError(f"bad parent entry at flat index {rc - 1}")
    return vis


def _common(case, vis=None, use_parent=None):
    """Argument tuple for the C functions. Mask input: parent unless ``vis`` is given."""
    dt = 0 if case.dtype == "f32" else 1
    arrs = [np.ascontiguousarray(x) for x in (case.q_nope, case.q_pe, case.c_kv, case.k_pe)]
    prefix = np.ascontiguousarray(case.prefix_len, dtype=np.int32)
    if vis is not None:
        parent = None
        vis = np.ascontiguousarray(vis, dtype=np.uint32)
    else:
        parent = np.ascontiguousarray(case.parent, dtype=np.int32)
    keep = arrs + [prefix, parent, vis]
    args = [case.B, case.T, case.H, dt] + [_ptr(a) for a in arrs] + [
        int(case.L), _ptr(prefix), _ptr(parent), _ptr(vis), float(case.scale)]
    return args, keep


def verify_attn(case, vis=None, nthreads: int = 0):
    """Whole problem. Returns (out float32 [B,T,H,512], lse float32 [B,T,H])."""
    args, keep = _common(case, vis)
    out = np.empty((case.B, case.T, case.H, 512), dtype=np.float32)
    lse = np.empty((case.B, case.T, case.H), dtype=np.float32)
    rc = _load().kdt_ref_verify_attn(*args, _ptr(out), _ptr(lse), int(nthreads))
    if rc:
        raise OracleError(f"oracle rejected the case (code {rc})")
    del keep
    return out, lse


def verify_attn_rows(case, rows, vis=None, nthreads: int = 0, f64: bool = False):
    """Selected flat rows r = (b*T + i)*H + h. Returns (out [n,512], lse [n]),
    float32 (rounded to nearest) or, with ``f64``, double."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    args, keep = _common(case, vis)
    n = rows.shape[0]
    if f64:
        out = np.empty((n, 512), dtype=np.float64)
        lse = np.empty(n, dtype=np.float64)
        ptrs = [None, None, _ptr(out), _ptr(lse)]
    else:
        out = np.empty((n, 512), dtype=np.float32)
        lse = np.empty(n, dtype=np.float32)
        ptrs = [_ptr(out), _ptr(lse), None, None]
    rc = _load().kdt_ref_verify_attn_rows(*args, _ptr(rows), n, *ptrs, int(nthreads))
    if rc:
        raise OracleError(f"oracle rejected the case (code {rc})")
    del keep
    return out, lse


def attn_weights(case, row: int, vis=None) -> np.ndarray:
    """Softmax weights (double) of flat row ``row`` over cache rows j < L."""
    args, keep = _common(case, vis)
    p = np.zeros(case.L, dtype=np.float64)
    rc = _load().kdt_ref_attn_weights(*args, int(row), _ptr(p))
    if rc:
        raise OracleError(f"oracle rejected the case (code {rc})")
    del keep
    return p


def merge_states(o_a, lse_a, o_b, lse_b):
    """Log-sum-exp merge of two attention states over disjoint key sets (double)."""
    o_a = np.ascontiguousarray(o_a, dtype=np.float64)
    o_b = np.ascontiguousarray(o_b, dtype=np.float64)
    lse_a = np.ascontiguousarray(lse_a, dtype=np.float64).reshape(-1)
    lse_b = np.ascontiguousarray(lse_b, dtype=np.float64).reshape(-1)
    n = lse_a.shape[0]
    D = o_a.size // max(n, 1)
    o = np.empty_like(o_a)
    lse = np.empty_like(lse_a)
    _load().kdt_ref_merge_states(n, D, _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o), _ptr(lse))
    return o, lse
