"""Multi-process (gloo, world size 2, CPU) checks of the bench's rank logic.

The decode path has no data-path collective: under torchrun every rank runs its
own replica of the workload, and the only exchange is the host-side maximum of
the per-rank times. These tests run that logic as two CPU processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(w)
    bench.barrier(dist)
    slowest = bench.reduce_max(dist, 1.0 + rank * 0.5)  # rank 1 is the slow one
    value = bench.aggregate_throughput(units_per_rank=300.0, world=w, max_seconds=slowest)
    # the reference arm runs on rank 0 only; other ranks return without work
    ref = bench.run_reference(None, w, r) if r != 0 else "rank0"
    dist.destroy_process_group()
    results[rank] = (slowest, value, ref)


def test_two_ranks_take_the_max_time_and_scale_weakly():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(results)
    assert res[0][0] == res[1][0] == pytest.approx(1.5)
    assert res[0][1] == res[1][1] == pytest.approx(300.0 * 2 / 1.5)
    assert res[1][2] is None


def test_single_process_helpers_without_torch_distributed():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.init_dist(1) is None
    assert bench.reduce_max(None, 3.25) == 3.25
    assert bench.aggregate_throughput(10.0, 1, 2.0) == 5.0
    assert bench.summarize_clocks([["0", "2070", "2070", "900", "0x0", "Not Active", "Not Active",
                                    "Not Active", "Active"]]) == {
        "sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 1, "reasons": ["sw_power_cap"]}
