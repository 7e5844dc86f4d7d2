"""The multi-GPU reporting path of bench.py on CPU: two gloo ranks, as torchrun starts
them, each with its own timings. Every rank must see the slowest rank's times, and the
whole-job value is the work of all ranks over that time (weak scaling, no collective on
the data path -- each rank runs its own copy of the workload)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.0 + rank, 0.5 + 2.0 * rank]        # rank 1 is slower on both
        got = bench.max_over_ranks(local, dist, torch.device("cpu"))
        queue.put((rank, got, bench.whole_job_tflops(1e12, world, got[0])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict()
    for _ in range(2):
        rank, got, value = q.get(timeout=120)
        res[rank] = (got, value)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank in (0, 1):
        got, value = res[rank]
        assert got == [2.0, 2.5]
        # 1e12 FLOP per rank, two ranks, slowest 2 ms: 1 PFLOP/s
        assert value == pytest.approx(1000.0)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], None, None) == [3.0, 4.0]
    assert bench.whole_job_tflops(2e12, 1, 4.0) == pytest.approx(500.0)
