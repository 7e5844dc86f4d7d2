"""Seeded synthetic inputs for tree-verify MLA-absorb attention.

This module produces random data and nothing else: normal draws, bf16 rounding of
those draws, random draft-tree parent arrays, prefix lengths and NaN padding. It
holds none of the attention arithmetic (no scores, no masks, no softmax, no
visibility bits), so both the CUDA path and the CPU oracle can take their inputs
from it without sharing any of the method.

Random numbers come from splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based generator:
element n of a stream keyed ``k`` is ``mix64(k + (n + 1) * 0x9E3779B97F4A7C15)``.
Uniforms take the top 53 bits; normals use the Box-Muller transform on
consecutive uniform pairs. Every tensor slice (tensor name, sequence b) has its
own stream, so a slice does not depend on how many other slices were drawn.

Workload shapes follow the benchmark configurations of the DDTree verify-attn
kernel (latent 512 + rope 64, scale 1/sqrt(192)); see ``CONFIGS``.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import numpy as np

D_C = 512   # latent (kv_lora) width of the MLA cache
D_R = 64    # rope width
SCALE = 1.0 / math.sqrt(192.0)

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BF16_NAN = np.uint16(0x7FC0)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, tag: str) -> np.uint64:
    t = np.array([zlib.crc32(tag.encode()) & 0xFFFFFFFF], dtype=np.uint64)
    s = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix64(s ^ _mix64(t))[0]


def raw_u64(seed: int, tag: str, n: int) -> np.ndarray:
    """First ``n`` outputs of the splitmix64 stream keyed by (seed, tag)."""
    key = _stream_key(seed, tag)
    idx = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * _GAMMA)


def uniform(seed: int, tag: str, n: int) -> np.ndarray:
    """``n`` doubles uniform on [0, 1) from the top 53 bits of each draw."""
    return (raw_u64(seed, tag, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tag: str, n: int, sigma: float = 1.0) -> np.ndarray:
    """``n`` doubles ~ N(0, sigma^2) by Box-Muller on uniform pairs."""
    m = (n + 1) // 2
    u = uniform(seed, tag, 2 * m)
    u1 = 1.0 - u[0::2]              # (0, 1]: log is finite
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n] * sigma


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round doubles to bfloat16 once, round-to-nearest-even, as uint16 bit patterns.

    Works on the float64 bit pattern directly (53-bit significand -> 8 bits), so
    there is no intermediate float32 rounding. Valid for finite inputs inside the
    bf16 normal range, which is all this module draws.
    """
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = (b + (np.uint64((1 << 44) - 1) + lsb)) & ~np.uint64((1 << 45) - 1)
    f32 = b.view(np.float64).astype(np.float32)     # exact: value has 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly (for display and host-side checks)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------------
# Draft-tree parent arrays. parent[0] = -1 (the root is tree query 0) and
# -1 <= parent[i] < i, so node order is topological.
# ----------------------------------------------------------------------------------

def tree_uniform(seed: int, tag: str, T: int, window: Optional[int] = None) -> np.ndarray:
    """parent[i] uniform in [max(0, i - window), i) (window None: [0, i))."""
    u = uniform(seed, tag, T)
    p = np.empty(T, dtype=np.int32)
    p[0] = -1
    for i in range(1, T):
        lo = 0 if window is None else max(0, i - window)
        p[i] = lo + min(int(u[i] * (i - lo)), i - lo - 1)
    return p


def tree_geometric(seed: int, tag: str, T: int, q: float = 0.5) -> np.ndarray:
    """Best-first-shaped tree: parent[i] = i - 1 - min(k, i - 1), k ~ Geometric(q) on {0,1,..}."""
    u = uniform(seed, tag, T)
    p = np.empty(T, dtype=np.int32)
    p[0] = -1
    for i in range(1, T):
        uu = 1.0 - u[i]                          # (0, 1]
        k = int(math.floor(math.log(uu) / math.log(1.0 - q)))
        p[i] = i - 1 - min(k, i - 1)
    return p


def tree_bounded_depth(seed: int, tag: str, T: int, max_depth: int = 16) -> np.ndarray:
    """parent[i] uniform over {j < i : depth(j) < max_depth}, depth(root) = 1."""
    u = uniform(seed, tag, T)
    p = np.empty(T, dtype=np.int32)
    depth = np.zeros(T, dtype=np.int64)
    p[0] = -1
    depth[0] = 1
    for i in range(1, T):
        cand = np.nonzero(depth[:i] < max_depth)[0]
        j = int(cand[min(int(u[i] * len(cand)), len(cand) - 1)])
        p[i] = j
        depth[i] = depth[j] + 1
    return p


def tree_chain(T: int) -> np.ndarray:
    p = np.arange(-1, T - 1, dtype=np.int32)
    return p


def tree_star(T: int) -> np.ndarray:
    p = np.zeros(T, dtype=np.int32)
    p[0] = -1
    return p


TREE_KINDS = {
    "uniform": lambda s, tag, T: tree_uniform(s, tag, T),
    "window8": lambda s, tag, T: tree_uniform(s, tag, T, window=8),
    "geometric": lambda s, tag, T: tree_geometric(s, tag, T),
    "depth16": lambda s, tag, T: tree_bounded_depth(s, tag, T, 16),
    "chain": lambda s, tag, T: tree_chain(T),
    "star": lambda s, tag, T: tree_star(T),
}


# ----------------------------------------------------------------------------------
# Cases
# ----------------------------------------------------------------------------------

@dataclasses.dataclass
class Case:
    """One verify-attn problem in host memory.

    Layouts (row-major): q_nope [B,T,H,512], q_pe [B,T,H,64], c_kv [B,L,512],
    k_pe [B,L,64]; float32 arrays when dtype == "f32", uint16 bf16 bit patterns
    when dtype == "bf16". Tree node t of sequence b sits at cache row
    prefix_len[b] + t; rows [prefix_len[b] + T, L) are padding filled with NaN.
    """
    name: str
    B: int
    T: int
    H: int
    L: int
    dtype: str
    q_nope: np.ndarray
    q_pe: np.ndarray
    c_kv: np.ndarray
    k_pe: np.ndarray
    prefix_len: np.ndarray     # int32 [B]
    parent: np.ndarray         # int32 [B,T]
    scale: float = SCALE
    vis_input: str = "parent"  # "parent": pass parent[]; "bits": pass packed bits built from it
    seed: int = 0

    @property
    def W(self) -> int:
        return (self.T + 31) // 32

    @property
    def kv_len(self) -> np.ndarray:
        return self.prefix_len.astype(np.int64) + self.T

    @property
    def max_kv_len(self) -> int:
        return int(self.kv_len.max())

    @property
    def rows(self) -> int:
        return self.B * self.T * self.H

    def nbytes(self) -> int:
        return sum(a.nbytes for a in (self.q_nope, self.q_pe, self.c_kv, self.k_pe,
                                      self.prefix_len, self.parent))


def _draw(seed, tag, n, sigma, dtype):
    x = normal(seed, tag, n, sigma)
    if dtype == "bf16":
        return f64_to_bf16_bits(x)
    return x.astype(np.float32)


def make_case(name: str, B: int, T: int, H: int, prefix, dtype: str = "f32",
              tree="uniform", sigma: float = 1.0, seed: int = 1, outlier_frac: float = 0.0,
              outlier_scale: float = 8.0, vis_input: str = "parent", L: Optional[int] = None,
              pad_value: str = "nan", scale: float = SCALE) -> Case:
    """Build a seeded case.

    ``prefix``: an int (all sequences) or a sequence of B ints, or a tuple
    ("uniform", lo, hi) for per-sequence prefixes uniform on [lo, hi].
    ``tree``: a TREE_KINDS key, or an int32 array [T] / [B,T] of parents.
    ``outlier_frac``: per cache row Bernoulli probability that the row's c_kv and
    k_pe are multiplied by ``outlier_scale`` (applied before bf16 rounding).
    """
    assert dtype in ("f32", "bf16")
    if isinstance(prefix, tuple) and prefix and prefix[0] == "uniform":
        lo, hi = int(prefix[1]), int(prefix[2])
        u = uniform(seed, "prefix", B)
        prefix_len = np.array([lo + min(int(x * (hi - lo + 1)), hi - lo) for x in u], dtype=np.int32)
    elif np.isscalar(prefix):
        prefix_len = np.full(B, int(prefix), dtype=np.int32)
    else:
        prefix_len = np.asarray(prefix, dtype=np.int32).reshape(B)
    kv_len = prefix_len.astype(np.int64) + T
    if L is None:
        L = int(kv_len.max())
    assert L >= int(kv_len.max())

    if isinstance(tree, str):
        parent = np.stack([TREE_KINDS[tree](seed, f"tree/{b}", T) for b in range(B)]).astype(np.int32)
    else:
        parent = np.asarray(tree, dtype=np.int32)
        if parent.ndim == 1:
            parent = np.broadcast_to(parent, (B, T)).copy()
    assert parent.shape == (B, T)

    store = np.uint16 if dtype == "bf16" else np.float32
    q_nope = np.empty((B, T, H, D_C), dtype=store)
    q_pe = np.empty((B, T, H, D_R), dtype=store)
    c_kv = np.empty((B, L, D_C), dtype=store)
    k_pe = np.empty((B, L, D_R), dtype=store)
    for b in range(B):
        q_nope[b] = _draw(seed, f"q_nope/{b}", T * H * D_C, sigma, dtype).reshape(T, H, D_C)
        q_pe[b] = _draw(seed, f"q_pe/{b}", T * H * D_R, sigma, dtype).reshape(T, H, D_R)
        n = int(kv_len[b])
        ck = normal(seed, f"c_kv/{b}", n * D_C, sigma).reshape(n, D_C)
        kp = normal(seed, f"k_pe/{b}", n * D_R, sigma).reshape(n, D_R)
        if outlier_frac > 0:
            hit = uniform(seed, f"outlier/{b}", n) < outlier_frac
            ck[hit] *= outlier_scale
            kp[hit] *= outlier_scale
        if dtype == "bf16":
            c_kv[b, :n] = f64_to_bf16_bits(ck)
            k_pe[b, :n] = f64_to_bf16_bits(kp)
        else:
            c_kv[b, :n] = ck.astype(np.float32)
            k_pe[b, :n] = kp.astype(np.float32)
        fill = (_BF16_NAN if dtype == "bf16" else np.float32(np.nan)) if pad_value == "nan" else 0
        c_kv[b, n:] = fill
        k_pe[b, n:] = fill
    return Case(name=name, B=B, T=T, H=H, L=L, dtype=dtype, q_nope=q_nope, q_pe=q_pe,
                c_kv=c_kv, k_pe=k_pe, prefix_len=prefix_len, parent=parent, scale=scale,
                vis_input=vis_input, seed=seed)


# The benchmark configurations. Seeds are 1000 + position in this table.
CONFIGS = {
    # B=2 H=8 prefix 37, T=9 (kv_len 46), fp32, parent uniform in [0, i)
    "tiny": dict(B=2, T=9, H=8, prefix=37, dtype="f32", tree="uniform", sigma=1.0),
    # Kimi-K2-shaped single decode verify, fp32, parent uniform in [max(0, i-8), i)
    "kimi": dict(B=1, T=32, H=64, prefix=4096, dtype="f32", tree="window8", sigma=1.0),
    # batched ragged verify, bf16, prefixes uniform in [1024, 8192], geometric tree
    "ragged": dict(B=8, T=64, H=64, prefix=("uniform", 1024, 8192), dtype="bf16",
                   tree="geometric", sigma=1.0),
    # H=64, 8K prefix, 64-node tree: every sequence at the top of the ragged range
    "target": dict(B=8, T=64, H=64, prefix=8192, dtype="bf16", tree="geometric", sigma=1.0),
    # long-context verify: sigma 0.5, 1% of cache rows scaled x8, depth <= 16
    "long": dict(B=4, T=128, H=64, prefix=32768, dtype="bf16", tree="depth16", sigma=0.5,
                 outlier_frac=0.01, outlier_scale=8.0),
    # DeepSeek-V3-shaped wide-head verify, visibility passed as packed bits
    "dsv3": dict(B=16, T=64, H=128, prefix=("uniform", 4096, 16384), dtype="bf16",
                 tree="uniform", sigma=1.0, vis_input="bits"),
}
CONFIG_SEEDS = {name: 1000 + k for k, name in enumerate(CONFIGS)}


def make_config(name: str, seed: Optional[int] = None, **overrides) -> Case:
    kw = dict(CONFIGS[name])
    kw.update(overrides)
    return make_case(name, seed=CONFIG_SEEDS[name] if seed is None else seed, **kw)


def config_shape(name: str) -> dict:
    """Shape of a configuration without drawing it (prefixes drawn, nothing else)."""
    kw = CONFIGS[name]
    B, T = kw["B"], kw["T"]
    prefix = kw["prefix"]
    seed = CONFIG_SEEDS[name]
    if isinstance(prefix, tuple):
        lo, hi = int(prefix[1]), int(prefix[2])
        u = uniform(seed, "prefix", B)
        pl = np.array([lo + min(int(x * (hi - lo + 1)), hi - lo) for x in u], dtype=np.int64)
    else:
        pl = np.full(B, int(prefix), dtype=np.int64)
    return dict(B=B, T=T, H=kw["H"], dtype=kw["dtype"], prefix_len=pl)


def random_vis_bits(seed: int, tag: str, B: int, T: int, density: float = 0.5,
                    force_self: bool = True) -> np.ndarray:
    """Arbitrary (not tree-shaped) packed visibility words [B,T,ceil(T/32)], bits >= T zero.

    Bit t (word t // 32, bit t % 32, LSB first) set means tree key t is visible.
    """
    W = (T + 31) // 32
    u = uniform(seed, tag, B * T * T).reshape(B, T, T)
    m = u < density
    if force_self:
        idx = np.arange(T)
        m[:, idx, idx] = True
    words = np.zeros((B, T, W), dtype=np.uint32)
    for t in range(T):
        words[:, :, t // 32] |= (m[:, :, t].astype(np.uint32) << np.uint32(t % 32))
    return words
