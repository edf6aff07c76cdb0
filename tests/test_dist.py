"""bench.py's multi-process logic on the CPU: world size 2 over gloo.

The path needs no data exchange between GPUs (every rank runs its own
replica of the step); the only collective is the max-over-ranks of the timed
region, which these ranks check with different per-rank times.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import torch.distributed as dist
    r, local, w = bench.dist_setup()
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w)          # ranks report 1.5 and 2.5
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_world2_gloo():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (0, 0, 1)
    assert bench.max_over_ranks(3.0, 1) == 3.0


def test_clock_sampler_keeps_only_the_timed_window(tmp_path):
    import bench
    p = tmp_path / "c.csv"
    p.write_text("2026/12/02 10:00:00.000, 0, 1000, 2070, 500, Active, Not Active, Not Active, "
                 "Not Active, Active\n"
                 "2026/12/02 10:00:01.000, 0, 1900, 2070, 900, Not Active, Not Active, Not Active, "
                 "Not Active, Not Active\n"
                 "2026/12/02 10:00:02.000, 0, 1950, 2070, 900, Not Active, Not Active, Not Active, "
                 "Not Active, Not Active\n")
    import datetime as dt
    t0 = dt.datetime(2026, 12, 2, 10, 0, 0, 500000).timestamp()
    t1 = dt.datetime(2026, 12, 2, 10, 0, 2, 500000).timestamp()
    r = bench.ClockSampler.summarize(str(p), t0, t1)
    assert r["sm_mhz"] == 1925.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == [] and r["samples_in_timed_region"] == 2 and r["samples_total"] == 3
