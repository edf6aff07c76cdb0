"""One step of the path (quantize-and-append, then attention) captured in a CUDA
graph and replayed.  Every replay must leave the pool equal, byte for byte, to
the oracle's pool after the same append, and give attention output within the
tolerance of the oracle's attention over that pool -- and, on the same inputs,
the same bits as eager launches.

Both entry points allocate nothing and hold no state between calls (the
attention's merge counters return to zero inside every launch), so a captured
step is reusable as long as the caller's buffers stay where they are.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, assert_close, require_gpu

pytestmark = pytest.mark.gpu


def _clear_slots(pages, slots):
    """Zero the K and V rows of the given slots (every kv-head)."""
    sl = torch.from_numpy(np.asarray(slots)).cuda()
    pages[sl // 16, :, :, sl % 16, :] = 0


def _capture(step):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                     # sizes the workspace before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


@pytest.mark.parametrize("num_splits", [0, 3])
def test_captured_verify_step_matches_the_oracle(num_splits):
    """The long-context stress step: an append chunk into a fragmented pool
    (offset 7 inside its first page), then the q_len 5 verify."""
    pq = require_gpu()
    w = W.workload("e4m3_verify_512k_stress", scale=0.004)
    c = Case(w, with_oracle=True)
    ak, av = W.append_chunk(w, "cuda")
    slots = torch.from_numpy(c.plan.append_slots).cuda()
    ws = pq.Workspace("cuda")
    out = torch.empty_like(c.q)

    def step():
        pq.kv_append_quant(ak, av, slots, w.kv_dtype, c.ks, c.vs, c.pages)
        pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                           num_splits=num_splits, workspace=ws, max_seq_len=max(w.seq_lens))

    g = _capture(step)
    eager_out = out.clone()
    pool = oracle.kv_append_quant(ak.cpu().numpy(), av.cpu().numpy(), c.plan.append_slots,
                                  w.kv_dtype, c.oracle_ks, c.oracle_vs, c.pool_o)
    ref = oracle.paged_attention(c.q.cpu().numpy(), pool, c.plan.block_table, w.seq_lens,
                                 w.q_len, w.kv_dtype, c.oracle_ks, c.oracle_vs)
    for i in range(2):
        out.fill_(float("nan"))
        _clear_slots(c.pages, c.plan.append_slots)     # the replay must write them again
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(c.gpu_pool_bytes(), pool), "replay %d: pool differs" % i
        assert_close(out, ref, "replay %d splits %d" % (i, num_splits))
        assert torch.equal(out, eager_out)


def test_captured_int8_decode_step_appends_and_attends():
    """The INT8 decode step: each replay appends the newest token of every
    sequence (per-kv-head scales) and runs q_len 1 attention over the grown
    cache.  The pool starts one token short per sequence, so the first replay
    is the real append; later replays rewrite the same codes."""
    pq = require_gpu()
    w = W.workload("int8_decode_append_262k", scale=0.004)
    kd, H = w.kv_dtype, w.num_kv_heads
    plan = W.plan_pool(w)
    ks, vs = W.calibrated_scales(w, "cuda")
    ks_np, vs_np = ks.cpu().numpy(), vs.cpu().numpy()
    pages = pq.new_pages(plan.num_pages, H, kd, "cuda", fill=0)
    pool = oracle.new_pool(plan.num_pages, H, 128, kd)
    for s, L in enumerate(w.seq_lens):
        sl = W.slots_for(plan, s, 0, L - 1)
        k, v = W.kv_tokens(w, s, 0, L - 1, "cuda")
        pq.kv_append_quant(k, v, torch.from_numpy(sl).cuda(), kd, ks, vs, pages)
        pool = oracle.kv_append_quant(k.cpu().numpy(), v.cpu().numpy(), sl, kd, ks_np, vs_np, pool)
    sk, sv, ssl = W.step_tokens(w, plan, "cuda")
    sslots = torch.from_numpy(ssl).cuda()
    q = W.query(w, "cuda")
    bt = torch.from_numpy(plan.block_table).cuda()
    lens = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    ws = pq.Workspace("cuda")
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        pq.kv_append_quant(sk, sv, sslots, kd, ks, vs, pages, status=status)
        pq.paged_attention(q, pages, bt, lens, 1, kd, ks, vs, out, workspace=ws, status=status,
                           max_seq_len=max(w.seq_lens))

    g = _capture(step)
    # the warm-up call before capture appended too: start one token short again
    _clear_slots(pages, ssl)
    pool = oracle.kv_append_quant(sk.cpu().numpy(), sv.cpu().numpy(), ssl, kd, ks_np, vs_np, pool)
    ref = oracle.paged_attention(q.cpu().numpy(), pool, plan.block_table, w.seq_lens, 1, kd,
                                 ks_np, vs_np)
    for i in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(pages.cpu().numpy(), pool), "replay %d: pool differs" % i
        assert_close(out, ref, "int8 decode replay %d" % i)
    assert int(status.item()) == 0


def test_captured_one_segment_fp16_decode_replays_like_the_oracle():
    """The tiny FP16 decode (one segment over 8 blocks, launched as a
    thread-block cluster that merges in shared memory) captured in a graph:
    several replays, each equal to the eager launch and within tolerance of
    the oracle."""
    pq = require_gpu()
    c = Case(W.workload("tiny_fp16_decode"))
    w = c.w
    ref = c.oracle_attention()
    eager = c.attention()
    out = torch.full_like(c.q, float("nan"))

    def step():
        pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                           max_seq_len=max(w.seq_lens))

    g = _capture(step)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
        assert_close(out, ref, "tiny decode, graph replay")
