#!/usr/bin/env python3
"""Benchmark of tree-verify MLA-absorb attention on GB300 (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch: one kdt_verify_attn call with
the parent array -- packed visibility bits, then scores, mask, online softmax, P.V,
split merge, epilogue (the tensor kernel overlaps the bits' kernel and waits for it
only before its first tree keys). Inputs are resident in HBM; L2 is flushed (256 MiB
write) between steps outside the timed events.

Workload: the H=64, 8K-prefix, 64-node-tree configuration -- B=8, H=64, every
prefix 8192, T=64 geometric-bias tree, bf16 q/c_kv/k_pe, fp32 out + lse -- seeded
synthetic data (``workloads``). ``--config`` selects another configuration.

The ``e2e`` figure times the same work end to end through kdt_verify_attn_host:
pinned host inputs in, host out and lse back, the copies pipelined with the compute.

One GPU only: the tensor-core kernel loads key tiles with cluster-multicast TMA,
which this library issues only over the memory of the one GPU a call runs on.
``--gpus N`` with N > 1 (or a torchrun launch with WORLD_SIZE > 1) prints one
``unavailable`` line on rank 0 and exits before any CUDA work.

``--impl reference`` times the CPU oracle as it stands on the host cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "verify-attn µs/call, TFLOP/s and KV GB/s at H=64; fraction of roofline"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
FP32_LANES_PER_SM = 128

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# dominant kernel from an ncu capture, keyed by kernel family and workload, with the
# hash of the kernel source it was taken on; reported only while that source is
# unchanged.
TRAFFIC = {
    ("tcgen05", "target"): {"src_hash": "2b8913615f321a79", "bytes": 156.91e6},
    ("tcgen05", "ragged"): {"src_hash": "2b8913615f321a79", "bytes": 155.58e6},
    ("tcgen05", "long"): {"src_hash": "2b8913615f321a79", "bytes": 338.96e6},
    ("tcgen05", "dsv3"): {"src_hash": "2b8913615f321a79", "bytes": 594.74e6},
    ("simt", "kimi"): {"src_hash": "31869aea57861729", "bytes": 14.31e6},
    ("simt_small", "tiny"): {"src_hash": "31869aea57861729", "bytes": 0.57e6},
    ("vc_proj", "target"): {"src_hash": "6d2fd9c107be75b7", "bytes": 77.55e6},
}


def single_gpu_only(gpus, world):
    """The unavailable line for a multi-GPU request, or None for one GPU."""
    n = max(gpus, world)
    if n <= 1:
        return None
    return {"metric": METRIC, "n_gpus": n,
            "unavailable": "one GPU per call: the tensor-core kernel's cluster-multicast TMA loads are "
                           "issued only over the memory of the GPU a call runs on, so no multi-GPU run exists"}


def fp32_fma_peak_tflops(sms, sm_mhz):
    """fp32 FMA roof: SMs x 128 lanes x 2 FLOP x SM clock."""
    return sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def kernel_src_hash(impl):
    import hashlib
    csrc = os.path.join(ROOT, "speculative_decoding_tree_absorb_gb300", "csrc")
    files = {"tcgen05": ["verify_tc.cu", "tc_ptx.cuh"], "vc_proj": ["vc_proj.cu", "tc_ptx.cuh"]}.get(
        impl, ["verify_simt.cu"])
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(impl, config):
    t = TRAFFIC.get((impl, config))
    if not t or t["src_hash"] != kernel_src_hash(impl):
        return None
    return t["bytes"]


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    except Exception:
        d = dict(FALLBACK)
        d["source"] = "fallback"
        return d


def depths(parent_row):
    d = np.zeros(len(parent_row), dtype=np.int64)
    for i, p in enumerate(parent_row):
        d[i] = 1 if p < 0 else d[p] + 1
    return d


def workload_counts(case):
    """Algorithmic FLOPs and bytes of one call (visible keys only; exps not counted)."""
    vis_keys = 0
    for b in range(case.B):
        vis_keys += int(case.prefix_len[b]) * case.T + int(depths(case.parent[b]).sum())
    flops = 2.0 * (wl.D_C + wl.D_C + wl.D_R) * case.H * vis_keys
    elt = 2 if case.dtype == "bf16" else 4
    kv_bytes = float(sum(int(k) for k in case.kv_len) * (wl.D_C + wl.D_R) * elt)
    rows = case.B * case.T * case.H
    q_bytes = rows * (wl.D_C + wl.D_R) * elt
    out_bytes = rows * wl.D_C * 4 + rows * 4
    meta = case.B * 4 + case.B * case.T * 4 + case.B * case.T * case.W * 4
    return dict(flops=flops, kv_bytes=kv_bytes, bytes=kv_bytes + q_bytes + out_bytes + meta, visible_keys=vis_keys)


class ClockSampler:
    """nvidia-smi clocks during the timed region (the query fields of the profiling recipe)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def make_workload(name):
    case = wl.make_config(name)
    return case


def run_reference(args, case, counts):
    """Time the CPU oracle on a bounded sample of the workload (rows of sequence 0)."""
    import oracle
    oracle.build()
    nthreads = oracle.num_threads()
    per_row_flops = counts["flops"] / case.rows
    # calibrate: a few rows, then size a sample for about --ref-seconds of CPU work
    rows = np.arange(min(16, case.rows))
    t0 = time.perf_counter()
    oracle.verify_attn_rows(case, rows)
    t_cal = time.perf_counter() - t0
    n = int(min(case.rows, max(len(rows), len(rows) * args.ref_seconds / max(t_cal, 1e-6) / max(1, args.steps))))
    n = max(1, n)
    sample = np.arange(n)
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle.verify_attn_rows(case, sample[: min(n, 8)])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.verify_attn_rows(case, sample)
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    flops = per_row_flops * n
    tflops = flops / sec / 1e12
    desc = f"first {n} rows (b=0, queries 0..{(n - 1) // case.H}, all heads) of the workload per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(args.config), "sample_rows": n},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle", "sample": desc},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def run_tree_ops(args, case, dev):
    """Time the steps next to verify on this workload's shapes: best-first tree build from
    synthetic drafter candidates (depth 16, 8 per depth, T - 1 nodes), NeoX RoPE in place
    on a combined [B,T,H,576] query buffer and the tree's key rows, greedy accept, and
    compaction of the accepted rows. CUDA events around each call, L2 flushed before each."""
    import torch
    import speculative_decoding_tree_absorb_gb300 as kdt

    def conv(x):
        if case.dtype == "bf16":
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(x).to(dev)

    B, T, H = case.B, case.T, case.H
    D, K, N = 16, 8, T - 1
    lp = -np.abs(wl.normal(77, "bench_lp", B * D * K)).reshape(B, D, K).astype(np.float32)
    ctok = (wl.raw_u64(77, "bench_tok", B * D * K) % 160000).astype(np.int32).reshape(B, D, K)
    ctok_d, lp_d = torch.from_numpy(ctok).to(dev), torch.from_numpy(lp).to(dev)
    comb = torch.cat([conv(case.q_nope), conv(case.q_pe)], dim=-1).contiguous()
    c_kv, k_pe = conv(case.c_kv), conv(case.k_pe)
    prefix = torch.from_numpy(case.prefix_len.astype(np.int32)).to(dev)
    parent, tok, depth, _ = kdt.tree_build(ctok_d, lp_d, N)
    pos = (prefix[:, None] + depth).to(torch.int32)
    target = torch.from_numpy((wl.raw_u64(77, "bench_tgt", B * T) % 2).astype(np.int32).reshape(B, T)).to(dev)
    tok = torch.remainder(tok, 2).to(torch.int32)                 # two-token alphabet: paths of a few nodes
    acc, n_acc, _ = kdt.tree_accept(parent, tok, target)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    esz = 2 if case.dtype == "bf16" else 4
    ops = {
        "tree_build": (lambda: kdt.tree_build(ctok_d, lp_d, N), B * D * K * 8 + 4 * B * T * 4, "latency"),
        "rope_neox": (lambda: kdt.rope_neox(pos, q=comb[..., 512:], k_pe=k_pe, prefix_len=prefix),
                      2 * (B * T * H + B * T) * 64 * esz, "fp64"),
        "tree_accept": (lambda: kdt.tree_accept(parent, tok, target), 3 * B * T * 4 + B * T * 4 + 8 * B, "latency"),
        "kv_compact": (lambda: kdt.kv_compact(c_kv, k_pe, prefix, acc, n_acc, update_prefix=False),
                       None, "latency"),
    }
    moved = int((n_acc - 1).clamp(min=0).sum().item())
    peaks = load_peaks()
    res = {}
    for name, (fn, nbytes, bound) in ops.items():
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        times = []
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1) * 1e3)
        if nbytes is None:
            nbytes = 2 * moved * (512 + 64) * esz
        us = statistics.mean(times)
        res[name] = {"us": us, "us_median": statistics.median(times), "bytes": nbytes,
                     "gbs": nbytes / (us * 1e-6) / 1e9, "frac_hbm": nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
                     "bound": bound}
    res["rope_neox"]["fp64_flops"] = 6 * (B * T * H + B * T) * 32
    return {"metric": "tree-step op time", "unit": "us", "higher_is_better": False, "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "dtype": "bf16" if case.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": workload_name(args.config), "B": B, "H": H, "T": T,
                       "builder": {"depth": D, "per_depth": K, "nodes": N}, "accepted_rows_moved": moved,
                       "l2": "flushed before each call"},
            "ops": res, "hbm_peak_gbs": peaks["hbm_gbs"]}


def run_vc_proj(args, case, dev):
    """Time the per-head w_vc up-projection (kdt_vc_up_proj) on this workload's verify
    output shape: o fp32 [B*T, H, 512] -> v fp32 [B*T, H, D_v] with bf16 weights
    [H, 512, D_v], D_v = 128. Synthetic N(0, 1) rows and N(0, 1/512) weights; CUDA events
    around each call on its stream, L2 flushed before each. HBM-bound: the roof is the
    algorithmic bytes (o read once, the weights once, v written once) at the measured
    copy bandwidth."""
    import torch
    import speculative_decoding_tree_absorb_gb300 as kdt
    R, H, D_v = case.B * case.T, case.H, 128
    o = torch.from_numpy(wl.normal(91, "bench_vc_o", R * H * 512).reshape(R, H, 512).astype(np.float32)).to(dev)
    wb = wl.f64_to_bf16_bits(wl.normal(91, "bench_vc_w", H * 512 * D_v, 1.0 / math.sqrt(512.0)))
    w = torch.from_numpy(wb.reshape(H, 512, D_v).view(np.int16)).view(torch.bfloat16).to(dev)
    v = torch.empty((R, H, D_v), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        kdt.vc_up_proj(o, w, out=v, err=err)
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0
    times = []
    with ClockSampler(dev.index or 0) as clk:
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            kdt.vc_up_proj(o, w, out=v, err=err)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1) * 1e3)
    assert int(err.item()) == 0
    peaks = load_peaks()
    nbytes = R * H * 512 * 4 + H * 512 * D_v * 2 + R * H * D_v * 4
    flops = 2.0 * R * H * 512 * D_v
    us = statistics.mean(times)
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"metric": "w_vc up-projection time", "value": us, "unit": "us", "higher_is_better": False, "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "dtype": "f32 rows x bf16 weights (fp32-accurate)",
            "data": "synthetic",
            "config": {"workload": f"{args.config} verify output: R={R} rows (B*T), H={H}, D_c=512, D_v={D_v}",
                       "l2": "flushed before each call"},
            "us_median": statistics.median(times), "tflops": flops / (us * 1e-6) / 1e12,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": measured_traffic("vc_proj", args.config),
                         "peak_basis": f"copy bandwidth ({peaks['source']})", "kernel": "vc_proj_kernel"},
            "algorithmic": {"bytes": nbytes, "flops": flops,
                            "roofline_us": nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6},
            "clocks": clk.summary(), "gpu_launches": args.steps}


def workload_name(name):
    d = wl.CONFIGS[name]
    pre = d["prefix"]
    pre_s = f"U[{pre[1]},{pre[2]}]" if isinstance(pre, tuple) else str(pre)
    return (f"{name}: B={d['B']} H={d['H']} prefix={pre_s} T={d['T']} {d['dtype']} "
            f"tree={d['tree']} latent=512 rope=64 scale=1/sqrt(192)")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kdt", choices=["kdt", "reference"])
    ap.add_argument("--config", default="target", choices=list(wl.CONFIGS))
    ap.add_argument("--kernel-impl", default="auto", choices=["auto", "simt", "tcgen05"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--ref-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="chunks kdt_verify_attn_host cuts the end-to-end step into (a divisor of B; "
                         "default 4, else 2, else 1)")
    ap.add_argument("--tree-ops", action="store_true",
                    help="time the steps around verify (tree build, RoPE, accept, compaction) instead")
    ap.add_argument("--vc-proj", action="store_true",
                    help="time the per-head w_vc up-projection of the verify output instead")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        case = make_workload(args.config)
        counts = workload_counts(case)
        print(json.dumps(run_reference(args, case, counts)), flush=True)
        return 0

    multi = single_gpu_only(args.gpus, world)
    if multi is not None:
        if rank == 0:
            print(json.dumps(multi), flush=True)
        return 0

    import torch
    import speculative_decoding_tree_absorb_gb300 as kdt
    from speculative_decoding_tree_absorb_gb300 import build_lib

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    torch.cuda.set_device(local_rank)
    build_lib.build()
    kdt.lib()

    case = make_workload(args.config)
    counts = workload_counts(case)
    dev = torch.device("cuda", local_rank)
    if args.tree_ops:
        print(json.dumps(run_tree_ops(args, case, dev)), flush=True)
        return 0
    if args.vc_proj:
        print(json.dumps(run_vc_proj(args, case, dev)), flush=True)
        return 0

    def conv(x):
        if case.dtype == "bf16":
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(x)

    host = dict(q_nope=conv(case.q_nope), q_pe=conv(case.q_pe), c_kv=conv(case.c_kv), k_pe=conv(case.k_pe),
                prefix_len=torch.from_numpy(case.prefix_len.astype(np.int32)),
                parent=torch.from_numpy(case.parent.astype(np.int32)))
    d = {k: v.to(dev) for k, v in host.items()}
    B, T, H = case.B, case.T, case.H
    W = case.W
    out = torch.empty((B, T, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # one call per step: the visibility bits from the parent array (in the workspace), then
    # the attention -- the tensor kernel starts while the bits are still being built
    a = kdt.make_args(d["q_nope"], d["q_pe"], d["c_kv"], d["k_pe"], d["prefix_len"], parent=d["parent"],
                      max_kv_len=case.max_kv_len, scale=case.scale, out=out, lse=lse, err=err,
                      impl=args.kernel_impl, num_splits=args.num_splits)
    pl = kdt.plan(a)
    ws = torch.empty(max(1, pl["workspace_bytes"]), dtype=torch.uint8, device=dev)
    lib = kdt.lib()
    import ctypes
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    ws_ptr = ctypes.c_void_p(ws.data_ptr())
    ws_n = ws.numel()
    launches_per_step = pl["num_launches"]

    def step():
        st = lib.kdt_verify_attn(ctypes.byref(a), ws_ptr, ws_n, sptr)
        if st != 0:
            raise kdt.KdtError(st, "kdt_verify_attn")

    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, "malformed tree reported"

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            e0, e1 = ev[k]
            e0.record(stream)
            st = lib.kdt_verify_attn(ctypes.byref(a), ws_ptr, ws_n, sptr)
            e1.record(stream)
            if st:
                raise kdt.KdtError(st, "timed step")
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    clocks = clk.summary()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    ms = statistics.mean(step_ms)
    # the attention call is the whole step: visibility bits, attention, piece merge
    ms_attn = ms
    ms_attn_median = statistics.median(step_ms)

    # ---- end to end through the C ABI with host buffers ------------------------------
    # kdt_verify_attn_host: pinned host tensors in, host out and lse back. The library cuts
    # the batch into chunks of whole sequences and overlaps each chunk's copy in, compute and
    # copy out on three streams (the host link, not the kernels, sets the pace).
    pinned = {k_: v.contiguous().pin_memory() for k_, v in host.items()}
    out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    n_chunks = args.e2e_chunks or next(c for c in (4, 2, 1) if B % c == 0)
    if n_chunks < 1 or B % n_chunks:
        raise SystemExit("--e2e-chunks must divide B")
    ah = kdt.make_args(pinned["q_nope"], pinned["q_pe"], pinned["c_kv"], pinned["k_pe"], pinned["prefix_len"],
                       parent=pinned["parent"], max_kv_len=case.max_kv_len, scale=case.scale, out=out_h, lse=lse_h,
                       err=err, impl=args.kernel_impl, num_splits=args.num_splits)
    dev_n = kdt.host_buffer_size(ah, n_chunks)
    if dev_n == 0:
        raise SystemExit("kdt_verify_attn_host rejected the arguments")
    dev_buf = torch.empty(dev_n, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    host_streams = [ctypes.c_void_p(x.cuda_stream) for x in (stream, s_in, s_out)]
    dev_ptr = ctypes.c_void_p(dev_buf.data_ptr())

    def e2e_step():
        st = lib.kdt_verify_attn_host(ctypes.byref(ah), n_chunks, dev_ptr, dev_n, *host_streams)
        if st != 0:
            raise kdt.KdtError(st, "kdt_verify_attn_host")

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms, enq_ms = [], []
    for _ in range(max(3, min(args.steps, 10))):
        flush.fill_(1)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_step()
        enq_ms.append((time.perf_counter() - t0) * 1e3)
        torch.cuda.synchronize(dev)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    # the host copy of the chunked run against the device-timed call on the same inputs: the
    # work splits differ (and with them the bf16 rounding of P). Each run is held to the
    # path's tolerance against the oracle, so the two may differ by up to twice that.
    e2e_out = out_h
    ref_out = out.cpu()
    tol = 2e-2 if case.dtype == "bf16" else 1e-4
    e2e_diff = (e2e_out - ref_out).abs()
    if bool((e2e_diff > 2 * (tol + tol * ref_out.abs())).any()):
        raise SystemExit(f"end-to-end output differs from the device-timed call by {e2e_diff.max().item()}")
    e2e_check = {"max_abs_diff": e2e_diff.max().item(), "mean_abs_diff": e2e_diff.mean().item()}
    e2e_mean = statistics.mean(e2e_ms)

    flops = counts["flops"]
    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_peak = fp32_fma_peak_tflops(sms, peaks.get("sm_max_mhz", 2070.0))
    tflops = flops / (ms * 1e-3) / 1e12
    attn_tflops = flops / (ms_attn * 1e-3) / 1e12
    if pl["impl"] == "tcgen05":
        peak = peaks["bf16_tflops"]
        bound, peak_note = "tensor", f"bf16 dense, cuBLAS burst ({peaks['source']})"
    else:
        peak = fp32_peak
        bound, peak_note = "alu", f"fp32 FMA: {sms} SMs x 128 lanes x 2 FLOP x max SM clock"
    # the workload's compute roof: bf16 inputs may use the tensor cores; fp32 inputs need
    # fp32 arithmetic (TF32 would not meet the fp32 tolerance), so the fp32 FMA peak
    if case.dtype == "bf16":
        compute_peak, compute_basis = peaks["bf16_tflops"], "bf16 tensor"
    else:
        compute_peak, compute_basis = fp32_peak, "fp32 FMA"
    compute_roof_us = flops / (compute_peak * 1e12) * 1e6
    hbm_roof_us = counts["bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e6
    roof_us = max(compute_roof_us, hbm_roof_us)

    cpu_baseline = None
    if not args.no_cpu_baseline:
        ref_args = argparse.Namespace(steps=1, warmup=0, ref_seconds=args.ref_seconds, config=args.config,
                                      gpus=1)
        r = run_reference(ref_args, case, counts)
        cpu_baseline = dict(r["cpu_baseline"])

    line = {
        "metric": METRIC,
        "value": tflops,
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if case.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": workload_name(args.config), "B": B, "H": H, "T": T,
                   "prefix": [int(x) for x in case.prefix_len[:4]] + (["..."] if B > 4 else []),
                   "kernel_impl": pl["impl"], "num_splits": pl["num_splits"],
                   "l2": "flushed between steps (256 MiB write outside the timed events)",
                   "parallelism": "one GPU"},
        "us_per_call": ms * 1e3,
        "us_per_call_attention": ms_attn * 1e3,
        "us_per_call_attention_median": ms_attn_median * 1e3,
        "tflops_attention": attn_tflops,
        "kv_gbs": counts["kv_bytes"] / (ms_attn * 1e-3) / 1e9,
        "workload_roofline": {"roofline_us": roof_us, "compute_us": compute_roof_us, "hbm_us": hbm_roof_us,
                              "frac": roof_us / (ms * 1e3), "basis": f"max(FLOPs/{compute_basis} peak, bytes/HBM) of "
                                                                    f"{peaks['source']} peaks"},
        "roofline": {"bound": bound, "achieved": attn_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak, "traffic": measured_traffic(pl["impl"], args.config),
                     "peak_basis": peak_note,
                     "kernel": f"verify_{pl['impl']} call: visibility bits, attention, piece/split merge"},
        "algorithmic": {"flops": flops, "bytes": counts["bytes"], "kv_bytes": counts["kv_bytes"]},
        "clocks": clocks,
        "e2e": {"value": flops / (e2e_mean * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_mean, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": f"kdt_verify_attn_host: {n_chunks} chunks of {B // n_chunks} sequence(s); copy in, "
                            f"compute and copy out on three streams",
                "host_enqueue_ms": statistics.mean(enq_ms), "vs_device_call": e2e_check},
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cpu_baseline,
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
