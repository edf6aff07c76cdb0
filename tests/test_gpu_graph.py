"""One step of the path (quantize-and-append, then verify attention) captured
in a CUDA graph and replayed: the replays must give what eager launches give.

Both entry points allocate nothing and hold no state between calls (the
attention's merge counters return to zero inside every launch), so a captured
step is reusable as long as the caller's buffers stay where they are.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import Case, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num_splits", [0, 3])
def test_captured_step_replays_like_eager(num_splits):
    pq = require_gpu()
    w = W.workload("e4m3_verify_512k_stress", scale=0.004)
    c = Case(w, with_oracle=False)
    ak, av = W.append_chunk(w, "cuda")
    slots = torch.from_numpy(c.plan.append_slots).cuda()
    ws = pq.Workspace("cuda")
    out = torch.empty_like(c.q)

    def step():
        pq.kv_append_quant(ak, av, slots, w.kv_dtype, c.ks, c.vs, c.pages)
        pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                           num_splits=num_splits, workspace=ws, max_seq_len=max(w.seq_lens))

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                     # sizes the workspace before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager_out = out.clone()
    eager_pages = c.pages.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager_out)
        assert torch.equal(c.pages, eager_pages)
