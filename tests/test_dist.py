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
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
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


def _dcp_rank(rank, world, port, out):
    """One CPU rank of a decode context parallel split: the oracle attends over
    this rank's page-aligned share of every sequence's keys, the ranks
    all-gather (O / l, lse) over gloo, and every rank merges."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    from tests.test_oracle_attention import _random_case
    from tests.test_oracle_dcp import shares
    dist.init_process_group("gloo")
    rng = np.random.default_rng(31)                      # same data on every rank
    q, pool, bt, L, ks, vs = _random_case(rng, [45, 70, 9], 2, 4, 16, 5, 1)
    bounds = [(0, 2), (2, 8)][rank:rank + 1]
    (lbt, ls, qp), = shares(bt, L, 5, bounds)
    o, lse = oracle.paged_attention_partial(q, pool, lbt, ls, qp, 5, 1, ks, vs)
    go = [torch.zeros(o.shape, dtype=torch.float64) for _ in range(world)]
    gl = [torch.zeros(lse.shape, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(go, torch.from_numpy(o))
    dist.all_gather(gl, torch.from_numpy(lse))
    merged, _ = oracle.merge_lse([x.numpy() for x in go], [x.numpy() for x in gl])
    full = oracle.paged_attention(q, pool, bt, L, 5, 1, ks, vs)
    out[rank] = float(np.abs(merged - full).max())
    dist.destroy_process_group()


def test_dcp_split_over_two_gloo_ranks_equals_full_attention():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_dcp_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    assert set(out.keys()) == {0, 1} and max(out.values()) < 1e-12
