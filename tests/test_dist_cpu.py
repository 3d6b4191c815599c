"""The multi-rank path of bench.py on the CPU: two gloo ranks.

Each rank runs bench's own helpers (environment, process group, barrier,
max over ranks, whole-job throughput) as a torchrun launch would; no GPU.
"""
import os
import queue
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    dist = bench.init_dist(w, backend="gloo")
    try:
        bench.barrier(dist)
        ms = bench.max_over_ranks(dist, 10.0 + 5.0 * r)  # rank 1 is the slower one
        value = bench.aggregate_gbps(w, 1_000_000, 4, ms)
        out.put((r, w, local, ms, value, dist.get_backend()))
        bench.barrier(dist)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = []
    try:
        for _ in procs:
            results.append(out.get(timeout=120))
    except queue.Empty:
        pytest.fail("a rank did not report within 120 s")
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    results.sort()
    assert [r[0] for r in results] == [0, 1] and all(r[1] == 2 and r[2] == r[0] for r in results)
    assert all(r[3] == 15.0 and r[5] == "gloo" for r in results), "every rank sees the slowest rank's time"
    want = 2 * 1_000_000 * 4 / 15e-3 / 1e9
    assert all(abs(r[4] - want) < 1e-12 for r in results), "value counts both ranks' bytes over the slowest time"


def test_single_process_needs_no_group():
    import bench
    assert bench.init_dist(1) is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.aggregate_gbps(1, 2_000_000, 10, 4.0) == pytest.approx(5.0)
