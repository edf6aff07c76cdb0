"""Real decode steps: each appends one new token per sequence into the pool
and then runs the decode attention over the grown cache, on the INT8 decode
workload (per-kv-head scales, q_len 1) at a size the oracle finishes quickly.
After every step the pool must equal the oracle's byte for byte and the
attention output must match the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import assert_close, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["int8_decode_append_262k", "e4m3_decode_b8"])
def test_eight_decode_steps_grow_the_cache(name):
    pq = require_gpu()
    w = W.workload(name, scale=0.004 if name.startswith("int8") else 0.05)
    n_steps = 8
    kd, H = w.kv_dtype, w.num_kv_heads
    plan = W.plan_pool(w)
    ks, vs = W.calibrated_scales(w, "cuda")
    ks_np, vs_np = ks.cpu().numpy(), vs.cpu().numpy()
    pages = pq.new_pages(plan.num_pages, H, kd, "cuda", fill=0)
    pool = oracle.new_pool(plan.num_pages, H, 128, kd)
    for s, L in enumerate(w.seq_lens):          # all but the last n_steps tokens
        sl = W.slots_for(plan, s, 0, L - n_steps)
        k, v = W.kv_tokens(w, s, 0, L - n_steps, "cuda")
        pq.kv_append_quant(k, v, torch.from_numpy(sl).cuda(), kd, ks, vs, pages)
        pool = oracle.kv_append_quant(k.cpu().numpy(), v.cpu().numpy(), sl, kd, ks_np, vs_np,
                                      pool)
    q = W.query(w, "cuda")
    bt = torch.from_numpy(plan.block_table).cuda()
    out = torch.empty_like(q)
    for i in range(n_steps):
        lens = [L - n_steps + i + 1 for L in w.seq_lens]
        new = [W.kv_tokens(w, s, n - 1, n, "cuda") for s, n in enumerate(lens)]
        k = torch.cat([a for a, _ in new])
        v = torch.cat([b for _, b in new])
        sl = np.array([W.slots_for(plan, s, n - 1, n)[0] for s, n in enumerate(lens)],
                      dtype=np.int64)
        pq.kv_append_quant(k, v, torch.from_numpy(sl).cuda(), kd, ks, vs, pages)
        pq.paged_attention(q, pages, bt, torch.tensor(lens, dtype=torch.int32, device="cuda"),
                           1, kd, ks, vs, out)
        pool = oracle.kv_append_quant(k.cpu().numpy(), v.cpu().numpy(), sl, kd, ks_np, vs_np,
                                      pool)
        assert np.array_equal(pages.cpu().numpy(), pool), "step %d: pool differs" % i
        ref = oracle.paged_attention(q.cpu().numpy(), pool, plan.block_table, lens, 1, kd,
                                     ks_np, vs_np)
        assert_close(out, ref, "%s step %d" % (name, i))
