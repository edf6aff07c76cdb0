"""The library keeps no state between calls: two attention calls on two
streams with their own workspaces, running at the same time, give exactly what
they give one after the other."""
import pytest
import torch

import workloads as W
from tests.helpers import Case, require_gpu

pytestmark = pytest.mark.gpu


def test_concurrent_streams_with_own_workspaces():
    pq = require_gpu()
    a = Case(W.workload("e4m3_verify_512k_stress", scale=0.01), with_oracle=False)
    b = Case(W.workload("int8_row_verify_131k", scale=0.01), with_oracle=False)
    ref_a = a.attention(num_splits=0).clone()
    ref_b = b.attention(num_splits=0).clone()
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    wa, wb = pq.Workspace("cuda"), pq.Workspace("cuda")
    oa, ob = torch.empty_like(a.q), torch.empty_like(b.q)
    for _ in range(3):
        oa.fill_(float("nan"))
        ob.fill_(float("nan"))
        torch.cuda.synchronize()
        for c, s, wsp, o in ((a, sa, wa, oa), (b, sb, wb, ob)):
            with torch.cuda.stream(s):
                pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, c.w.q_len, c.w.kv_dtype, c.ks,
                                   c.vs, o, num_splits=0, workspace=wsp,
                                   max_seq_len=max(c.w.seq_lens), stream=s)
        torch.cuda.synchronize()
        assert torch.equal(oa, ref_a) and torch.equal(ob, ref_b)
