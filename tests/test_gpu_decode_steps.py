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


# the FP16 decode and the 32-row verify kernels may start early (programmatic
# dependent launch); the INT8 decode at this size runs the paired kernel,
# which does not
@pytest.mark.parametrize("name,scale", [("tiny_fp16_decode", 1.0), ("e4m3_verify_q8_131k", 0.004),
                                        ("int8_decode_append_262k", 0.004)])
def test_back_to_back_steps_see_the_tokens_just_appended(name, scale):
    """Every step's append is followed at once by its attention on the same
    stream (all inputs prepared beforehand, nothing else launched between), so
    the attention kernel may become resident while the append is running; it
    must still see every code the append writes.  The newest tokens' K rows
    are scaled up so that they carry much of the softmax weight."""
    pq = require_gpu()
    w = W.workload(name, scale=scale)
    n_steps = 6
    kd, H, ql = w.kv_dtype, w.num_kv_heads, w.q_len
    plan = W.plan_pool(w)
    ks, vs = W.calibrated_scales(w, "cuda")
    ks_np, vs_np = ks.cpu().numpy(), vs.cpu().numpy()
    pages = pq.new_pages(plan.num_pages, H, kd, "cuda", fill=0)
    pool = oracle.new_pool(plan.num_pages, H, 128, kd)
    per = ql                                       # tokens appended per sequence per step
    for s, L in enumerate(w.seq_lens):
        sl = W.slots_for(plan, s, 0, L - n_steps * per)
        k, v = W.kv_tokens(w, s, 0, L - n_steps * per, "cuda")
        pq.kv_append_quant(k, v, torch.from_numpy(sl).cuda(), kd, ks, vs, pages)
        pool = oracle.kv_append_quant(k.cpu().numpy(), v.cpu().numpy(), sl, kd, ks_np, vs_np,
                                      pool)
    q = W.query(w, "cuda")
    bt = torch.from_numpy(plan.block_table).cuda()
    steps = []
    for i in range(n_steps):
        lens = [L - (n_steps - 1 - i) * per for L in w.seq_lens]
        parts = [W.kv_tokens(w, s, n - per, n, "cuda") for s, n in enumerate(lens)]
        k = torch.cat([a for a, _ in parts]) * 3        # newest keys: larger scores
        v = torch.cat([b for _, b in parts])
        sl = np.concatenate([W.slots_for(plan, s, n - per, n) for s, n in enumerate(lens)])
        steps.append((k, v, torch.from_numpy(sl).cuda(),
                      torch.tensor(lens, dtype=torch.int32, device="cuda"), lens, sl))
    outs = [torch.empty_like(q) for _ in range(n_steps)]
    torch.cuda.synchronize()
    for i, (k, v, sl_d, lens_d, _, _) in enumerate(steps):
        pq.kv_append_quant(k, v, sl_d, kd, ks, vs, pages)
        pq.paged_attention(q, pages, bt, lens_d, ql, kd, ks, vs, outs[i],
                           max_seq_len=max(w.seq_lens))
    torch.cuda.synchronize()
    for i, (k, v, _, _, lens, sl) in enumerate(steps):
        pool = oracle.kv_append_quant(k.cpu().numpy(), v.cpu().numpy(), sl, kd, ks_np, vs_np,
                                      pool)
        ref = oracle.paged_attention(q.cpu().numpy(), pool, plan.block_table, lens, ql, kd,
                                     ks_np, vs_np)
        assert_close(outs[i], ref, "%s back-to-back step %d" % (name, i))
    got = pages.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if kd == W.FP16 else got.numpy()
    assert np.array_equal(got, pool)
