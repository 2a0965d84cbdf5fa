"""bench.py's multi-rank logic on CPU: gloo, world size 2.  Every rank runs an
independent replica; the timing collectives take the max of the elapsed
times and the sum of the work."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    bench.dist_init(world)
    m = bench.max_over_ranks(1.5 + rank, world)
    s = bench.sum_over_ranks(10.0 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, m, s))
    dist.destroy_process_group()


def test_timing_collectives_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda args: called.append(1))
    assert bench.main(["--impl", "reference"]) == 0
    assert not called


def test_clock_summary_window():
    import bench
    s = bench.ClockSampler("GPU-0")
    s.samples = [(10.0, 1500.0, 2070.0, []), (10.5, 1900.0, 2070.0, ["sw_power_cap"]),
                 (20.0, 300.0, 2070.0, ["hw_slowdown"])]
    out = s.summary(9.9, 11.0)
    assert out["sm_mhz"] == 1700.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 2
