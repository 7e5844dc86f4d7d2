"""Test-side helpers: golden-file parsing, library-routine references, tolerances.

The library references here use only torch CPU float64 primitives (matmul,
softmax, logsumexp) on explicit masks; they are the independent pins the oracle is
checked against, never the product path.
"""
from __future__ import annotations

import itertools
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Tolerances: |gpu - ref| <= ATOL + RTOL * |ref|, applied to out and lse.
TOL = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 2e-2)}


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored inputs -> float64, exactly."""
    if dtype == "bf16":
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def closure_visible(parent_row: np.ndarray) -> np.ndarray:
    """Boolean [T,T]: vis[i,t] iff t is i or an ancestor of i.

    Computed as the reflexive-transitive closure of the child->parent relation by
    repeated boolean matrix products (numpy matmul), not by walking pointers.
    """
    T = len(parent_row)
    A = np.zeros((T, T), dtype=np.int64)
    for i, p in enumerate(parent_row):
        if p >= 0:
            A[i, p] = 1
    R = np.eye(T, dtype=np.int64)
    for _ in range(T):
        R2 = ((np.eye(T, dtype=np.int64) + A @ R) > 0).astype(np.int64)
        if np.array_equal(R2, R):
            break
        R = R2
    return R.astype(bool)


def pack_bits(vis_bool: np.ndarray) -> np.ndarray:
    """Boolean [..., T] -> uint32 words [..., ceil(T/32)], bit t%32 of word t//32."""
    T = vis_bool.shape[-1]
    W = (T + 31) // 32
    out = np.zeros(vis_bool.shape[:-1] + (W,), dtype=np.uint32)
    for t in range(T):
        out[..., t // 32] |= vis_bool[..., t].astype(np.uint32) << np.uint32(t % 32)
    return out


def all_parent_arrays(T: int):
    """Every parent array with parent[0] = -1 and -1 <= parent[i] < i."""
    ranges = [range(-1, i) for i in range(1, T)]
    for combo in itertools.product(*ranges):
        yield np.array((-1,) + combo, dtype=np.int32)


def torch_reference(case, key_mask: np.ndarray):
    """Masked softmax attention in torch float64 (library matmul/softmax/logsumexp).

    key_mask: bool [B, T, kv] (kv = case.L) of visible keys per (b, i).
    Returns (out [B,T,H,512], lse [B,T,H]) as float64 numpy arrays.
    """
    import torch
    qn = torch.from_numpy(widen(case.q_nope, case.dtype))
    qp = torch.from_numpy(widen(case.q_pe, case.dtype))
    ck = torch.from_numpy(np.nan_to_num(widen(case.c_kv, case.dtype)))
    kp = torch.from_numpy(np.nan_to_num(widen(case.k_pe, case.dtype)))
    mask = torch.from_numpy(key_mask)
    outs, lses = [], []
    for b in range(case.B):
        s = case.scale * (torch.einsum("thd,kd->thk", qn[b], ck[b]) + torch.einsum("thd,kd->thk", qp[b], kp[b]))
        m = mask[b][:, None, :].expand_as(s)
        s = s.masked_fill(~m, float("-inf"))
        lse = torch.logsumexp(s, dim=-1)
        p = torch.softmax(s, dim=-1)
        p = torch.nan_to_num(p, nan=0.0)
        outs.append(torch.einsum("thk,kd->thd", p, ck[b]))
        lses.append(lse)
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


def tree_key_mask(case, vis_bool=None) -> np.ndarray:
    """bool [B,T,L]: prefix rows plus visible tree rows (from the closure or given bools)."""
    B, T, L = case.B, case.T, case.L
    mask = np.zeros((B, T, L), dtype=bool)
    for b in range(B):
        P = int(case.prefix_len[b])
        vb = closure_visible(case.parent[b]) if vis_bool is None else vis_bool[b]
        mask[b, :, :P] = True
        mask[b, :, P:P + T] = vb
    return mask


def read_golden_cases(fname: str):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest, "paths": {}}
                cases.append(cur)
            elif key == "prefix":
                cur["prefix"] = int(rest)
            elif key == "parent":
                cur["parent"] = np.array([int(x) for x in rest.split()], dtype=np.int32)
            elif key == "count":
                cur["count"] = [int(x) for x in rest.split()]
            elif key == "path":
                i, _, nodes = rest.partition(":")
                cur["paths"][int(i)] = [int(x) for x in nodes.split()]
    return cases


def assert_close(got, ref, atol, rtol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_inf = np.isinf(ref) & (got == ref)
    err = np.abs(got - ref)
    bad = ~(both_inf | (err <= atol + rtol * np.abs(ref)))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance "
            f"(atol={atol}, rtol={rtol}); max abs err {np.nanmax(np.where(both_inf, 0, err)):.3e}; "
            f"first {idx.tolist()} got {[got[tuple(i)] for i in idx]} ref {[ref[tuple(i)] for i in idx]}")
