"""Full-size workloads in the launch configuration bench.py times, checked on
sampled (sequence, kv-head) segments that the oracle computes one at a time.

The GPU side fills the whole pool with kv_append_quant and runs one bench step
(for the stress workload: the 8192-token append into the fragmented pool, then
the balanced split-KV verify).  The oracle side regenerates only the sampled
segment's K and V from the seeded generator, encodes them itself into a pool
of its own and runs its float64 attention; nothing it uses comes from the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, assert_close, require_gpu

pytestmark = pytest.mark.gpu

SAMPLES = {   # workload -> sampled (sequence, kv-head) segments
    "e4m3_verify_512k_stress": [(0, 3), (5, 6)],     # a 524288-token and a 32768-token sequence
    "e4m3_verify_131k": [(4, 1)],
    "int8_decode_append_262k": [(1, 2)],
    "e4m3_decode_b8": [(3, 5), (6, 0)],
    "int8_row_decode_262k": [(2, 7)],
    "int8_row_verify_131k": [(6, 4)],
    "e4m3_verify_q8_131k": [(2, 3)],                 # 32 query rows per kv-head
}


def _oracle_segment(w, q, s, h, ks, vs, window=0):
    """float64 output rows [q_len, G, D] of (sequence s, kv-head h)."""
    L = w.seq_lens[s]
    n = w.pages_of(L)
    k, v = W.kv_tokens(w, s, 0, L, "cpu", heads=[h])
    pool = oracle.new_pool(n, 1, w.head_dim, w.kv_dtype)
    if w.kv_dtype == W.INT8_ROW:           # scales come from the rows themselves
        pool, ks, vs = oracle.kv_append_quant(k.numpy(), v.numpy(), np.arange(L, dtype=np.int64),
                                              w.kv_dtype, oracle.new_scale_pool(n, 1),
                                              oracle.new_scale_pool(n, 1), pool)
    else:
        pool = oracle.kv_append_quant(k.numpy(), v.numpy(), np.arange(L, dtype=np.int64),
                                      w.kv_dtype, [ks], [vs], pool)
        ks, vs = [ks], [vs]
    G = w.group
    rows = q[s * w.q_len:(s + 1) * w.q_len, h * G:(h + 1) * G]
    return oracle.paged_attention(rows, pool, np.arange(n, dtype=np.int32)[None, :], [L],
                                  w.q_len, w.kv_dtype, ks, vs, window=window)


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_sampled_segments(name):
    pq = require_gpu()
    w = W.workload(name)
    c = Case(w, with_oracle=False)
    if w.append_tokens:
        plan = c.plan
        ak, av = W.append_chunk(w, "cuda")
        pq.kv_append_quant(ak, av, torch.from_numpy(plan.append_slots).cuda(), w.kv_dtype,
                           c.ks, c.vs, c.pages)
    out = c.attention(num_splits=0, max_seq_len=max(w.seq_lens)).float().cpu().numpy()
    q = c.q.cpu().numpy()
    ks_all, vs_all = c.ks.cpu().numpy(), c.vs.cpu().numpy()
    G = w.group
    for s, h in SAMPLES[name]:
        ks = float(ks_all[h if w.scale_per_head else 0])
        vs = float(vs_all[h if w.scale_per_head else 0])
        ref = _oracle_segment(w, q, s, h, ks, vs)
        got = out[s * w.q_len:(s + 1) * w.q_len, h * G:(h + 1) * G]
        assert_close(got, ref, "%s seq %d head %d" % (name, s, h))
    del c
    torch.cuda.empty_cache()


def test_full_size_sliding_window_sampled_segments():
    # the 131K verify with the 2048-token window bench.py times beside it
    pq = require_gpu()
    w = W.workload("e4m3_verify_131k")
    c = Case(w, with_oracle=False)
    out = torch.full_like(c.q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                       num_splits=0, window=2048, status=status, max_seq_len=max(w.seq_lens))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    out = out.float().cpu().numpy()
    q = c.q.cpu().numpy()
    G = w.group
    for s, h in [(1, 5), (7, 0)]:
        ref = _oracle_segment(w, q, s, h, float(c.ks.cpu()[0]), float(c.vs.cpu()[0]), window=2048)
        got = out[s * w.q_len:(s + 1) * w.q_len, h * G:(h + 1) * G]
        assert_close(got, ref, "window 2048 seq %d head %d" % (s, h))
    del c
    torch.cuda.empty_cache()
