"""bench.py runs on one GPU only: the tensor-core kernel issues cluster-multicast TMA
loads, which this library keeps to the memory of the GPU a call runs on. A multi-GPU
request (``--gpus N`` or a torchrun launch with WORLD_SIZE > 1) must end with one
``unavailable`` line on rank 0, nothing on the other ranks, exit status 0, and no CUDA
work -- these run on a CPU-only machine, so any CUDA call would fail them."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    e["CUDA_VISIBLE_DEVICES"] = ""
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          cwd=ROOT, env=e, timeout=300)


def test_gpus_flag_above_one_is_refused_before_cuda_work():
    r = _bench("--gpus", "2", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and "unavailable" in d and "multicast" in d["unavailable"]


def test_torchrun_ranks_are_refused_quietly_except_rank_zero():
    r0 = _bench("--gpus", "4", env={"RANK": "0", "LOCAL_RANK": "0", "WORLD_SIZE": "4"})
    r1 = _bench("--gpus", "4", env={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "4"})
    assert r0.returncode == 0 and r1.returncode == 0
    assert json.loads(r0.stdout.strip())["n_gpus"] == 4
    assert r1.stdout.strip() == ""


def test_one_gpu_request_is_not_refused():
    import bench
    assert bench.single_gpu_only(1, 1) is None
    assert bench.single_gpu_only(1, 2)["n_gpus"] == 2
    assert bench.fp32_fma_peak_tflops(152, 2070.0) == 152 * 128 * 2 * 2070e6 / 1e12
