"""CPU oracle for the steps around tree-verify attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module; the library never calls it and shares no code with it.
Plain numpy (float64) and Python loops, one function per step, each following its
definition as stated below.

Parity status per function (how each is pinned is in ``tests/test_oracle_tree_ops.py``):
  rope_neox        -- pinned (complex-exponential form of the rotation, identity at
                      position 0, norm preservation, scores depend only on the position
                      difference, rotation by p then q equals rotation by p + q)
  tree_positions   -- pinned (chain and star trees, depth from explicit paths)
  tree_accept      -- pinned (brute force over all root paths on random trees with
                      distinct sibling tokens; all-match chain; no-match root)
  kv_compact       -- pinned (identity on a chain path; rows compared one by one with
                      the rows the path names)
  tree_build       -- pinned (brute force: every node of the full K-ary candidate tree
                      sorted by the selection order, first N taken; path-score and depth
                      invariants; single-candidate chain)
  vc_up_proj       -- pinned (one-hot selection weights return the selected latent
                      dims exactly; a unit latent returns the named weight row; the
                      triangular closed forms n + 1 and n (n + 1) / 2 fix the summation
                      range; bf16 weights widen exactly)
"""
from __future__ import annotations

import heapq

import numpy as np


# ---------------------------------------------------------------- NeoX RoPE --
def rope_neox(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """NeoX rotary embedding ("The Query-Split Kernel: A Pivotal Edit ...", "Input
    Knowledge: What One Must Understand to Grasp This Edit": element j pairs with element
    j + d/2 and the pair turns by an angle that grows with the position, the angles in float64
    to match a numpy reference; the engine itself computes in float32, "The Architecture
    of an Inference Engine ...", "The Context: Building an Engine from Scratch").

    For a vector x of even width d (values exact in float32) at position p, and j < d/2:
        w_j = base ** (-2 j / d),  a_j = p * w_j                      (float64)
        c_j = fl32(cos a_j),  s_j = fl32(sin a_j)                       (float64, rounded once)
        y[j]       = fl32( fl32(x[j] c_j)       - fl32(x[j + d/2] s_j) )
        y[j + d/2] = fl32( fl32(x[j + d/2] c_j) + fl32(x[j] s_j) )
    every float32 product and sum rounded to nearest on its own (no fused multiply-add).
    x: array [..., d]; pos: integer array of shape x.shape[:-1] (or broadcastable).
    Returns float32 [..., d].
    """
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    if d % 2:
        raise ValueError("rope width must be even")
    half = d // 2
    j = np.arange(half, dtype=np.float64)
    w = np.power(float(base), -2.0 * j / d)                        # [half], float64
    a = np.asarray(pos, dtype=np.float64)[..., None] * w          # [..., half], float64
    c = np.cos(a).astype(np.float32)
    s = np.sin(a).astype(np.float32)
    x1, x2 = x[..., :half], x[..., half:]
    y = np.empty(x.shape, dtype=np.float32)
    y[..., :half] = (x1 * c) - (x2 * s)
    y[..., half:] = (x2 * c) + (x1 * s)
    return y


def tree_positions(parent: np.ndarray, prefix_len: np.ndarray) -> np.ndarray:
    """Rotary position of tree node i: prefix_len[b] + depth(i), depth(root) = 0 (the
    root is the token after the committed prefix and a node sits one step after its
    parent; the forward pass takes token ids with their positions, "The Architecture of
    an Inference Engine ...", "What the Message Actually Says").
    parent int [B,T] in topological order; returns int64 [B,T]."""
    parent = np.asarray(parent)
    B, T = parent.shape
    depth = np.zeros((B, T), dtype=np.int64)
    for b in range(B):
        for i in range(T):
            p = int(parent[b, i])
            depth[b, i] = 0 if p < 0 else depth[b, p] + 1
    return depth + np.asarray(prefix_len, dtype=np.int64)[:, None]


# ------------------------------------------------------- greedy tree accept --
def tree_accept(parent: np.ndarray, tok: np.ndarray, target: np.ndarray):
    """Greedy walk of a verified tree (the third Phase-1 kernel, a greedy walk deciding
    which draft tokens are accepted: "The Moment of Truth: Validating a Custom CUDA
    Attention Kernel ...", "Context: Building a Native DDTree Inference Engine").

    Node 0 is the root. tok[i] is node i's draft token, target[i] the target model's
    greedy next token after node i. From the root, repeatedly move to the child c of the
    current node with tok[c] == target[current] (the lowest such index if several);
    stop when there is none. Returns per sequence (path, bonus): the node indices from
    the root to the last accepted node, and target[last] (the token the target adds).
    parent/tok/target int [B,T]."""
    parent = np.asarray(parent)
    tok = np.asarray(tok)
    target = np.asarray(target)
    B, T = parent.shape
    res = []
    for b in range(B):
        path = [0]
        cur = 0
        while True:
            nxt = -1
            for c in range(T):
                if int(parent[b, c]) == cur and int(tok[b, c]) == int(target[b, cur]):
                    nxt = c
                    break
            if nxt < 0:
                break
            path.append(nxt)
            cur = nxt
        res.append((path, int(target[b, cur])))
    return res


def kv_compact(c_kv: np.ndarray, k_pe: np.ndarray, prefix_len: np.ndarray, paths):
    """Post-verify cache compaction (the cache is compacted after acceptance to drop the
    unaccepted branches: "The Architecture of an Inference Engine ...", "The Context:
    Building an Engine from Scratch" and "Input Knowledge Required"). The tree's rows sit
    at prefix_len[b] + t; the accepted path's k-th node moves to row prefix_len[b] + k,
    and the new prefix length is prefix_len[b] + len(path). Rows past the new length
    keep whatever they held. c_kv [B,L,Dc], k_pe [B,L,Dr] (any dtype, copied as stored).
    Returns (c_kv', k_pe', new_prefix_len)."""
    c2 = np.array(c_kv, copy=True)
    k2 = np.array(k_pe, copy=True)
    newp = np.array(prefix_len, dtype=np.int64, copy=True)
    for b, path in enumerate(paths):
        p0 = int(prefix_len[b])
        src_c = [np.array(c_kv[b, p0 + t]) for t in path]
        src_k = [np.array(k_pe[b, p0 + t]) for t in path]
        for k in range(len(path)):
            c2[b, p0 + k] = src_c[k]
            k2[b, p0 + k] = src_k[k]
        newp[b] = p0 + len(path)
    return c2, k2, newp


# ------------------------------------------------------- best-first builder --
def tree_build(cand_tok: np.ndarray, cand_lp: np.ndarray, N: int, root_tok=None):
    """Best-first draft tree ("The Architecture of an Inference Engine ...", section "The
    Context": a GPU best-first tree builder constructs the draft tree on the device,
    replacing a per-request CPU heap).

    The drafter gives, for every depth d = 1..D ahead of the root, K candidate tokens
    cand_tok[b, d-1, :] with log-probabilities cand_lp[b, d-1, :] (the same candidates
    below every node of depth d-1). A node's score is the float32 sum of the
    log-probabilities on its path (root 0). Starting from the root, the tree grows by the
    best node not yet in it whose parent is, N times. "Best" is the order: higher score,
    then lower depth, then lower parent index, then lower candidate rank, where a depth's
    candidates are ranked by log-probability, highest first, ties by position.
    Nodes are numbered in the order they join (root 0), so parents precede children.
    Returns int32 parent [B,N+1], tok [B,N+1] (tok[b,0] = root_tok[b] or -1), depth
    [B,N+1] and float32 score [B,N+1]."""
    cand_tok = np.asarray(cand_tok)
    cand_lp = np.asarray(cand_lp, dtype=np.float32)
    B, D, K = cand_lp.shape
    T = N + 1
    parent = np.full((B, T), -1, dtype=np.int32)
    tok = np.full((B, T), -1, dtype=np.int32)
    depth = np.zeros((B, T), dtype=np.int32)
    score = np.zeros((B, T), dtype=np.float32)
    for b in range(B):
        # rank of each candidate: log-probability descending, ties by position
        order = [sorted(range(K), key=lambda k: (-float(cand_lp[b, d, k]), k)) for d in range(D)]
        if root_tok is not None:
            tok[b, 0] = int(root_tok[b])
        heap = []

        def push(par, d, r):                         # candidate of rank r at depth d (1-based) under par
            k = order[d - 1][r]
            sc = np.float32(score[b, par] + cand_lp[b, d - 1, k])
            heapq.heappush(heap, (-float(sc), d, par, r, sc))

        if D > 0:
            for r in range(K):
                push(0, 1, r)
        for n in range(1, T):
            _, d, par, r, sc = heapq.heappop(heap)
            parent[b, n], depth[b, n], score[b, n] = par, d, sc
            tok[b, n] = int(cand_tok[b, d - 1, order[d - 1][r]])
            if d < D:
                for r2 in range(K):
                    push(n, d + 1, r2)
    return parent, tok, depth, score


# ---------------------------------------------------- value up-projection (w_vc) --
def vc_up_proj(o: np.ndarray, w_vc: np.ndarray, w_dtype: str = "bf16") -> np.ndarray:
    """Per-head value up-projection of the latent attention output ("The Verify-Attn
    Kernel: A Single File Write ...", "Design Decisions and Trade-Offs": the attention
    output stays in the latent space and the value projection of each head is its own
    GEMM afterwards, the split SGLang uses).

        v[..., h, n] = sum_{d < D_c} o[..., h, d] * w_vc[h, d, n]

    o: float32 [..., H, D_c] (the rows of a verify output, e.g. [B, T, H, 512]);
    w_vc: [H, D_c, D_v], bf16 bit patterns (uint16) when ``w_dtype`` is "bf16", else
    float32. Both are widened exactly to float64, each head's product is one float64
    matrix multiply, and the result is rounded once to float32 [..., H, D_v].
    """
    o64 = np.asarray(o, dtype=np.float32).astype(np.float64)
    if w_dtype == "bf16":
        w32 = (np.asarray(w_vc, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    else:
        w32 = np.asarray(w_vc, dtype=np.float32)
    w64 = w32.astype(np.float64)
    H, D_c, D_v = w64.shape
    if o64.shape[-2:] != (H, D_c):
        raise ValueError("o must end in [H, D_c] matching w_vc [H, D_c, D_v]")
    v = np.empty(o64.shape[:-1] + (D_v,), dtype=np.float64)
    for h in range(H):
        v[..., h, :] = o64[..., h, :] @ w64[h]
    return v.astype(np.float32)
