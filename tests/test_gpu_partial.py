"""Decode-context-parallel building blocks on the GPU: each "rank" (run in
turn on this one GPU -- no kernel waits on another) attends over its
page-aligned share of the keys with pqkv_paged_attention_partial, and
pqkv_lse_merge combines the shares.  Checked against the oracle's partial
results and against full attention."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, assert_close, require_gpu
from tests.test_oracle_dcp import shares

pytestmark = pytest.mark.gpu


def _run_shares(pq, c, bounds, num_splits):
    w = c.w
    L = list(w.seq_lens)
    outs = []
    for lbt, ls, qp in shares(c.plan.block_table, L, w.q_len, bounds):
        o = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")
        lse = torch.empty(c.q.shape[:2], dtype=torch.float32, device="cuda")
        pq.paged_attention_partial(c.q, c.pages, torch.from_numpy(lbt).cuda(),
                                   torch.from_numpy(ls.astype(np.int32)).cuda(),
                                   torch.from_numpy(qp.astype(np.int32)).cuda(), w.q_len,
                                   w.kv_dtype, c.ks, c.vs, o, lse, num_splits=num_splits)
        outs.append((o, lse, lbt, ls, qp))
    return outs


@pytest.mark.parametrize("name,bounds", [
    ("e4m3_verify_512k_stress", [(0, 40), (40, 200)]),          # the long sequences cut in two
    ("e4m3_verify_131k", [(0, 30), (30, 60), (60, 100)]),       # a share cuts the draft window
    ("int8_row_decode_262k", [(0, 10), (10, 200), (200, 300)]),  # the last share is empty
])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_shares_match_oracle_and_merge_to_full_attention(name, bounds, num_splits):
    pq = require_gpu()
    scale = {"e4m3_verify_512k_stress": 0.004, "e4m3_verify_131k": 0.01,
             "int8_row_decode_262k": 0.004}[name]
    c = Case(W.workload(name, scale=scale))
    w = c.w
    outs = _run_shares(pq, c, bounds, num_splits)
    q = c.q.cpu().numpy()
    for o, lse, lbt, ls, qp in outs:
        ro, rl = oracle.paged_attention_partial(q, c.pool_o, lbt, ls, qp, w.q_len, w.kv_dtype,
                                                c.oracle_ks, c.oracle_vs)
        assert_close(o.cpu().numpy(), ro, "%s share o" % name)
        gl = lse.cpu().numpy().astype(np.float64)
        assert np.array_equal(np.isneginf(gl), np.isneginf(rl))
        fin = np.isfinite(rl)
        if fin.any():
            assert np.abs(gl[fin] - rl[fin]).max() <= 1e-3 + 1e-5 * np.abs(rl[fin]).max()
    parts_o = torch.stack([x[0] for x in outs])
    parts_l = torch.stack([x[1] for x in outs])
    out = torch.empty_like(c.q)
    out_lse = torch.empty(c.q.shape[:2], dtype=torch.float32, device="cuda")
    pq.lse_merge(parts_o, parts_l, out, out_lse)
    assert_close(out, c.oracle_attention(), "%s merged" % name)
    whole = oracle.paged_attention_partial(q, c.pool_o, c.plan.block_table, np.array(w.seq_lens),
                                           np.array(w.seq_lens) - w.q_len, w.q_len, w.kv_dtype,
                                           c.oracle_ks, c.oracle_vs)[1]
    assert np.abs(out_lse.cpu().numpy() - whole).max() <= 1e-3 + 1e-5 * np.abs(whole).max()


def test_single_share_partial_equals_attention():
    pq = require_gpu()
    c = Case(W.workload("e4m3_verify_131k", scale=0.01), with_oracle=False)
    w = c.w
    o = torch.empty(c.q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(c.q.shape[:2], dtype=torch.float32, device="cuda")
    qp = (c.seq_lens - w.q_len).to(torch.int32)
    pq.paged_attention_partial(c.q, c.pages, c.bt, c.seq_lens, qp, w.q_len, w.kv_dtype, c.ks, c.vs,
                               o, lse)
    ref = c.attention().float()
    assert torch.allclose(o, ref, rtol=1e-2, atol=2e-3)
    merged = torch.empty_like(c.q)
    pq.lse_merge(o[None].contiguous(), lse[None].contiguous(), merged)
    assert torch.allclose(merged.float(), ref, rtol=1e-2, atol=2e-3)


@pytest.mark.parametrize("num_splits", [7, 64])
def test_shares_with_many_partitions(num_splits):
    pq = require_gpu()
    c = Case(W.workload("e4m3_verify_512k_stress", scale=0.004))
    outs = _run_shares(pq, c, [(0, 50), (50, 200)], num_splits)
    out = torch.empty_like(c.q)
    pq.lse_merge(torch.stack([x[0] for x in outs]), torch.stack([x[1] for x in outs]), out)
    assert_close(out, c.oracle_attention(), "many partitions %d" % num_splits)
