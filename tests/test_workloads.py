"""Host-side checks of the seeded input generator and pool planning."""
import numpy as np
import torch

import workloads as W


def test_values_are_deterministic_and_sliceable():
    a = W.draw_values(9, W.KIND_K, 3, 0, 300, 4, 128, True)
    b = W.draw_values(9, W.KIND_K, 3, 0, 300, 4, 128, True)
    assert torch.equal(a, b)
    c = W.draw_values(9, W.KIND_K, 3, 100, 200, [1, 2], 128, True)
    assert torch.equal(c, a[100:200, 1:3])
    d = W.draw_values_chunked(9, W.KIND_K, 3, 0, 300, 4, 128, True, "cpu", chunk=64)
    assert torch.equal(d, a)


def test_streams_differ_by_kind_seq_head():
    base = W.draw_values(1, W.KIND_K, 0, 0, 64, 1, 128, False)
    for other in [W.draw_values(1, W.KIND_V, 0, 0, 64, 1, 128, False),
                  W.draw_values(1, W.KIND_K, 1, 0, 64, 1, 128, False),
                  W.draw_values(1, W.KIND_K, 0, 0, 64, [1], 128, False),
                  W.draw_values(2, W.KIND_K, 0, 0, 64, 1, 128, False)]:
        assert (other != base).float().mean() > 0.99


def test_distribution_moments_and_outlier_rate():
    x = W.draw_values(4, W.KIND_K, 0, 0, 4096, 8, 128, False).float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    y = W.draw_values(4, W.KIND_K, 0, 0, 4096, 8, 128, True).float()
    frac = (y != x).float().mean().item()
    assert 0.008 < frac < 0.012
    assert torch.allclose(y[y != x], (x[y != x] * 20).half().float())


def test_hash_known_values_stable():
    # regression guard: the generator must not change silently
    h = W.hash32(torch.arange(4, dtype=torch.int64), 0).tolist()
    assert h == W.hash32(torch.arange(4, dtype=torch.int64), 0).tolist()
    assert all(0 <= v < 2 ** 32 for v in h) and len(set(h)) == 4


def test_workload_shapes():
    w = W.workload("tiny_fp16_decode")
    assert (w.seq_lens, w.num_q_heads, w.num_kv_heads, w.q_len, w.kv_dtype) == ([1024], 8, 1, 1, W.FP16)
    w = W.workload("e4m3_decode_b8")
    assert len(w.seq_lens) == 8 and all(2048 <= x <= 32768 for x in w.seq_lens)
    assert (w.num_q_heads, w.num_kv_heads, w.q_len) == (32, 8, 1)
    w = W.workload("e4m3_verify_131k")
    assert w.seq_lens == [131072] * 8 and w.q_len == 5 and w.kv_bytes() == 2147483648
    w = W.workload("int8_decode_append_262k")
    assert w.seq_lens == [262144] * 4 and w.kv_dtype == W.INT8 and w.scale_per_head
    w = W.workload("e4m3_verify_512k_stress")
    assert w.seq_lens == [524288] * 2 + [32768] * 6 and w.append_tokens == 8192
    assert w.kv_bytes() == 2550136832
    # the row-scaled INT8 pool also reads two fp16 scales per (token, kv-head)
    w = W.workload("int8_row_decode_262k")
    assert w.kv_bytes() == 4 * 262144 * 8 * (2 * 128 + 2 * 2)
    assert w.append_bytes(1) == 8 * (2 * 128 * 2 + 2 * 128 + 2 * 2) + 8


def test_plan_pool_is_a_valid_shuffled_assignment():
    w = W.workload("e4m3_verify_512k_stress", scale=0.01)
    plan = W.plan_pool(w)
    used = []
    for s, L in enumerate(w.seq_lens):
        n = w.pages_of(L)
        row = plan.block_table[s]
        assert (row[:n] >= 0).all() and (row[n:] == -1).all()
        used.extend(row[:n].tolist())
    chunk_pages = set((plan.append_slots // 16).tolist())
    assert len(set(used)) == len(used)
    assert not (chunk_pages & set(used))
    assert max(used + list(chunk_pages)) < plan.num_pages
    assert plan.append_slots[0] % 16 == 7
    assert len(np.unique(plan.append_slots)) == len(plan.append_slots)
    # consecutive logical pages are scattered
    assert np.mean(np.abs(np.diff(plan.block_table[0, :w.pages_of(w.seq_lens[0])])) == 1) < 0.1


def test_scales_follow_amax():
    w = W.workload("int8_decode_append_262k", scale=0.002)
    ks, vs = W.calibrated_scales(w)
    assert ks.shape == (8,) and vs.shape == (8,)
    k, _ = W.kv_tokens(w, 0, 0, w.seq_lens[0])
    amax0 = max(W.kv_tokens(w, s, 0, L)[0][:, 0].float().abs().max().item()
                for s, L in enumerate(w.seq_lens))
    assert ks[0].item() == np.float32(amax0 / 127.0)


def test_decode_step_tokens_are_the_newest_of_each_sequence():
    # the INT8 decode step appends one token per sequence: the last one of
    # each sequence, at the slot the block table gives it
    w = W.workload("int8_decode_append_262k", scale=0.004)
    plan = W.plan_pool(w)
    k, v, slots = W.step_tokens(w, plan)
    B, H = w.num_seqs, w.num_kv_heads
    assert k.shape == v.shape == (B, H, 128) and slots.shape == (B,)
    assert W.step_append_tokens(w) == B
    for s, L in enumerate(w.seq_lens):
        kk, vv = W.kv_tokens(w, s, L - 1, L)
        assert torch.equal(k[s], kk[0]) and torch.equal(v[s], vv[0])
        assert slots[s] == plan.block_table[s, (L - 1) // 16] * 16 + (L - 1) % 16
    stress = W.workload("e4m3_verify_512k_stress")
    assert W.step_append_tokens(stress) == 8192
