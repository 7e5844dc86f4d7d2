"""The attention kernels start while the visibility kernel of the same call still runs
(programmatic dependent launch) and the merge passes while the attention kernel ends.
That overlap must never reach back past the call: a kernel the caller queued just
before -- here one that rewrites the cache, the queries and the prefix lengths -- must
be complete before the call reads anything. Each case rewrites the inputs on the GPU
right before the call, in the same stream, and checks every element against the oracle
on the new inputs, for all three kernel families. A fuzz over random small shapes then
runs every kernel family against the oracle."""
import zlib

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


@pytest.mark.parametrize("impl,dtype", [("tcgen05", "bf16"), ("simt", "f32"), ("simt_small", "f32")])
def test_inputs_written_just_before_the_call_are_seen(kdt, oracle_mod, impl, dtype):
    import torch
    old = wl.make_case("before", B=2, T=24, H=64, prefix=(900, 1300), dtype=dtype, tree="geometric", seed=11)
    new = wl.make_case("after", B=2, T=24, H=64, prefix=(1000, 1250), dtype=dtype, tree="geometric", seed=12,
                       L=old.L)
    d_old, d_new = G.to_device(old), G.to_device(new)
    d = {k: v.clone() for k, v in d_old.items()}                 # the call's buffers hold the old case
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    side = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    for rep in range(3):
        side.fill_(rep)                                          # keep the GPU busy ahead of the copies
        for k in ("q_nope", "q_pe", "c_kv", "k_pe", "prefix_len", "parent"):
            d[k].copy_(d_new[k])                                 # kernels queued right before the call
        out, lse = kdt.verify_attn(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"],
                                   parent=d["parent"], max_kv_len=new.L, scale=new.scale, impl=impl, stream=stream)
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle_mod.verify_attn(new)
        H.assert_close(out.cpu().numpy(), ref_out, *H.TOL[dtype], what=f"{impl} out after rewrite")
        H.assert_close(lse.cpu().numpy(), ref_lse, *H.TOL[dtype], what=f"{impl} lse after rewrite")
        for k in ("q_nope", "q_pe", "c_kv", "k_pe", "prefix_len", "parent"):
            d[k].copy_(d_old[k])


@pytest.mark.parametrize("seed", range(12))
def test_random_small_shapes_all_kernels(kdt, oracle_mod, seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 5))
    T = int(rng.choice([1, 2, 5, 9, 17, 33, 64]))
    Hh = int(rng.choice([1, 3, 8, 16, 64]))
    prefix = tuple(int(x) for x in rng.integers(0, 700, size=B))
    tree = str(rng.choice(["uniform", "geometric", "chain", "star", "depth16", "window8"]))
    for dtype in ("f32", "bf16"):
        case = wl.make_case(f"fuzz{seed}", B=B, T=T, H=Hh, prefix=prefix, dtype=dtype, tree=tree,
                            seed=zlib.crc32(f"fuzz{seed}".encode()) % 1000)
        ref_out, ref_lse = oracle_mod.verify_attn(case)
        impls = ["simt", "simt_small"] + (["tcgen05"] if dtype == "bf16" else [])
        for impl in impls:
            out, lse, err = G.run(case, impl=impl)
            assert err == 0
            H.assert_close(out, ref_out, *H.TOL[dtype], what=f"fuzz {seed} {impl} {dtype} out")
            H.assert_close(lse, ref_lse, *H.TOL[dtype], what=f"fuzz {seed} {impl} {dtype} lse")
