"""paged_attention on the GPU against the float64 oracle.

Bar: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise, plus a relative L2
bound of 1e-2 (the absolute term alone would let near-uniform long-context
outputs pass trivially), and a "needle" variant that makes outputs O(1).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, assert_close, require_gpu

pytestmark = pytest.mark.gpu

SMALL = {  # context scale per workload: small enough for the oracle, several tiles + ragged tail
    "tiny_fp16_decode": 1.0,
    "e4m3_decode_b8": 0.05,
    "e4m3_verify_131k": 0.01,
    "int8_decode_append_262k": 0.004,
    "e4m3_verify_512k_stress": 0.004,
}

_cases = {}


def case(name):
    if name not in _cases:
        _cases[name] = Case(W.workload(name, scale=SMALL[name]))
    return _cases[name]


@pytest.mark.parametrize("name", W.WORKLOAD_NAMES)
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_small_workloads_match_oracle(name, num_splits):
    c = case(name)
    assert np.array_equal(c.gpu_pool_bytes(), c.pool_o)
    ref = c.oracle_attention()
    out = c.attention(num_splits=num_splits)
    assert_close(out, ref, "%s splits=%d" % (name, num_splits))


@pytest.mark.parametrize("splits", [2, 7, 64, 128])     # 128: the largest split count
def test_split_count_invariance(splits):
    c = case("e4m3_verify_512k_stress")
    a = c.attention(num_splits=1).float()
    b = c.attention(num_splits=splits).float()
    assert_close(b, a.cpu().numpy().astype(np.float64), "splits %d vs 1" % splits)


def test_bitwise_deterministic_and_page_order_invariant():
    c = case("e4m3_verify_131k")
    a = c.attention(num_splits=0)
    b = c.attention(num_splits=0)
    assert torch.equal(a, b)
    # move every page to a new place in the pool: the output must not change
    pq = require_gpu()
    perm = np.random.default_rng(9).permutation(c.plan.num_pages)      # new -> old
    inv = np.argsort(perm)
    pages2 = c.pages[torch.from_numpy(perm).cuda()].contiguous()
    bt2 = np.where(c.plan.block_table >= 0, inv[np.maximum(c.plan.block_table, 0)], -1)
    out = torch.empty_like(c.q)
    pq.paged_attention(c.q, pages2, torch.from_numpy(bt2.astype(np.int32)).cuda(), c.seq_lens,
                       c.w.q_len, c.w.kv_dtype, c.ks, c.vs, out, num_splits=0)
    assert torch.equal(out, a)


@pytest.mark.parametrize("kv_dtype", [W.FP16, W.FP8_E4M3, W.INT8, W.INT8_ROW])
@pytest.mark.parametrize("q_len,G", [(1, 1), (1, 4), (5, 4), (1, 8), (3, 8), (8, 2), (2, 12),
                                     (7, 4), (8, 4), (5, 6)])
def test_row_shapes(kv_dtype, q_len, G):
    # every padded-row width (8, 16, 24, 32) and ragged lengths, incl. L == q_len;
    # q_len 7 and 8 with G 4 are the wider speculative verify (28 and 32 rows)
    w = W.Workload("shape", 40 + q_len * 10 + G, [q_len, 17, 100, 333], 2 * G, 2, q_len, kv_dtype,
                   outliers=kv_dtype != W.FP16, pool_slack=0.3)
    c = Case(w)
    for ns in (0, 1, 2):
        assert_close(c.attention(num_splits=ns), c.oracle_attention(), "q_len %d G %d" % (q_len, G))


def test_needle_outputs_are_order_one():
    # every query row of a sequence is the same vector u; 8 keys per sequence
    # (two inside the draft window) are 3u for every kv-head, so they take most
    # of the softmax mass and the outputs are O(1) instead of ~1/sqrt(L).  The
    # edits are made from CPU data and applied to both pools.
    pq = require_gpu()
    w = W.workload("e4m3_verify_512k_stress", scale=0.004)
    c = Case(w)
    rng = np.random.default_rng(4)
    ks, vs = c.ks.cpu().numpy(), c.vs.cpu().numpy()
    q = c.q.cpu().clone()
    for s, L in enumerate(w.seq_lens):
        u = torch.from_numpy(rng.normal(0, 1, 128).astype(np.float16))
        q[s * w.q_len:(s + 1) * w.q_len] = u
        pos = np.concatenate([rng.choice(L - w.q_len, 6, replace=False), [L - 3, L - 1]])
        k0, v0 = W.kv_tokens(w, s, 0, L, "cpu")
        fk = k0[pos].clone()
        fk[:] = (u.float() * 3.0).half()
        fv = v0[pos].contiguous()
        slots = W.slots_for(c.plan, s, 0, L)[pos]
        c.pool_o = oracle.kv_append_quant(fk.numpy(), fv.numpy(), slots, w.kv_dtype, ks, vs, c.pool_o)
        pq.kv_append_quant(fk.cuda(), fv.cuda(), torch.from_numpy(slots).cuda(), w.kv_dtype,
                           c.ks, c.vs, c.pages)
    c.q = q.cuda()
    assert np.array_equal(c.gpu_pool_bytes(), c.pool_o)
    ref = c.oracle_attention()
    assert np.abs(ref).max() > 0.3
    for ns in (0, 1, 5):
        assert_close(c.attention(num_splits=ns), ref, "needle splits %d" % ns)


def test_every_e4m3_code_in_k_and_v():
    # K and V tiles filled with all 256 codes (NaN codes excluded): checks the
    # in-register widening of every code, subnormals and -0 included
    pq = require_gpu()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    L = 64
    num_pages = 4
    rng = np.random.default_rng(6)
    pool = np.zeros((num_pages, 1, 2, 16, 128), np.uint8)
    tok = rng.choice(codes, size=(L, 2, 128))
    for j in range(L):
        pool[j // 16, 0, 0, j % 16] = tok[j, 0]
        pool[j // 16, 0, 1, j % 16] = tok[j, 1]
    q = torch.from_numpy(rng.normal(0, 0.02, (1, 4, 128)).astype(np.float16)).cuda()
    bt = torch.tensor([[0, 1, 2, 3]], dtype=torch.int32, device="cuda")
    sl = torch.tensor([L], dtype=torch.int32, device="cuda")
    ks = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    vs = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    pq.paged_attention(q, torch.from_numpy(pool).cuda(), bt, sl, 1, W.FP8_E4M3, ks, vs, out)
    ref = oracle.paged_attention(q.cpu().numpy(), pool, bt.cpu().numpy(), [L], 1, W.FP8_E4M3,
                                 [0.01], [0.5])
    assert_close(out, ref, "all codes")


@pytest.mark.parametrize("kv_dtype", [W.INT8, W.INT8_ROW])
@pytest.mark.parametrize("q_len", [1, 5])
def test_every_int8_code_in_k_and_v(kv_dtype, q_len):
    # every byte value (-128 .. 127; append never writes -128, the widening
    # must still be exact) at many (token, dim) places of K and V, for both
    # 8-bit integer formats and both row widths (8 and 24 padded query rows)
    pq = require_gpu()
    L, num_pages = 64, 4
    rng = np.random.default_rng(7 + q_len)
    pool = np.zeros((num_pages, 1, 2, 16, 128), np.uint8)
    base = np.tile(np.arange(256, dtype=np.uint8), 64).reshape(L, 2, 128)
    tok = rng.permuted(base.reshape(-1)).reshape(L, 2, 128)   # each value exactly 64 times
    for j in range(L):
        pool[j // 16, 0, 0, j % 16] = tok[j, 0]
        pool[j // 16, 0, 1, j % 16] = tok[j, 1]
    G = 4
    # scores spread over a few units, so that a wrong K code moves the output
    q = torch.from_numpy(rng.normal(0, 0.5, (q_len, G, 128)).astype(np.float16)).cuda()
    bt = torch.tensor([[0, 1, 2, 3]], dtype=torch.int32, device="cuda")
    sl = torch.tensor([L], dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    if kv_dtype == W.INT8:
        pages = torch.from_numpy(pool).cuda()
        ks = torch.tensor([0.05], dtype=torch.float32, device="cuda")
        vs = torch.tensor([0.03], dtype=torch.float32, device="cuda")
        pq.paged_attention(q, pages, bt, sl, q_len, kv_dtype, ks, vs, out)
        ref = oracle.paged_attention(q.cpu().numpy(), pool, bt.cpu().numpy(), [L], q_len,
                                     kv_dtype, [0.05], [0.03])
    else:
        pages = pq.new_pages(num_pages, 1, W.INT8_ROW, "cuda", fill=0)
        pages.copy_(torch.from_numpy(pool))
        kp = rng.uniform(0.02, 0.08, (num_pages, 1, 16)).astype(np.float16)
        vp = rng.uniform(0.01, 0.05, (num_pages, 1, 16)).astype(np.float16)
        sc = pq.row_scales(pages)
        sc[:, :, 0].copy_(torch.from_numpy(kp).view(num_pages, 1, 2, 8))
        sc[:, :, 1].copy_(torch.from_numpy(vp).view(num_pages, 1, 2, 8))
        kp, vp = kp.astype(np.float32), vp.astype(np.float32)
        pq.paged_attention(q, pages, bt, sl, q_len, kv_dtype, None, None, out)
        ref = oracle.paged_attention(q.cpu().numpy(), pool, bt.cpu().numpy(), [L], q_len,
                                     kv_dtype, kp, vp)
    assert_close(out, ref, "all int8 codes, format %d, q_len %d" % (kv_dtype, q_len))


def test_stale_nan_codes_past_the_end_are_ignored():
    pq = require_gpu()
    w = W.Workload("nan_tail", 77, [37, 50], 8, 2, 5, W.FP8_E4M3, pool_slack=0.5)
    c = Case(w, with_oracle=True, fill=0x7F)     # every unwritten code is NaN
    assert_close(c.attention(num_splits=0), c.oracle_attention(), "NaN tail")


def test_out_of_range_page_id_reads_zeros_and_reports():
    pq = require_gpu()
    w = W.Workload("badpage", 78, [40], 4, 1, 1, W.INT8, pool_slack=0.5)
    c = Case(w)
    bt = c.bt.clone()
    bt[0, 1] = 10 ** 6
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(c.q)
    pq.paged_attention(c.q, c.pages, bt, c.seq_lens, 1, W.INT8, c.ks, c.vs, out, status=status)
    assert "block-table page id out of range" in pq.status_bits(status)
    pool = c.pool_o.copy()
    bt_np = c.plan.block_table.copy()
    spare = pool.shape[0]
    pool = np.concatenate([pool, np.zeros_like(pool[:1])])
    bt_np[0, 1] = spare
    ref = oracle.paged_attention(c.q.cpu().numpy(), pool, bt_np, w.seq_lens, 1, W.INT8,
                                 c.ks.cpu().numpy(), c.vs.cpu().numpy())
    assert_close(out, ref, "zero page")


def test_host_validation_errors():
    pq = require_gpu()
    c = case("tiny_fp16_decode")
    out = torch.empty_like(c.q)
    with pytest.raises(ValueError):
        pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, 2, W.FP16, c.ks, c.vs, out)
    with pytest.raises(ValueError):
        pq.paged_attention(c.q[:, :7], c.pages, c.bt, c.seq_lens, 1, W.FP16, c.ks, c.vs, out)
    q9 = torch.zeros((1, 9 * 8, 128), dtype=torch.float16, device="cuda")   # 72 rows per kv-head
    with pytest.raises(ValueError):
        pq.paged_attention(q9, c.pages, c.bt, c.seq_lens, 1, W.FP16, c.ks, c.vs, torch.empty_like(q9))


def test_host_tensors_rejected():
    # a host tensor's pointer must never reach a kernel: each entry point
    # refuses it before launching anything
    pq = require_gpu()
    c = case("e4m3_verify_131k")
    w = c.w
    out = torch.empty_like(c.q)
    args = dict(q=c.q, bt=c.bt, seq_lens=c.seq_lens, ks=c.ks, vs=c.vs, out=out)
    for name in args:
        bad = dict(args)
        bad[name] = args[name].cpu()
        with pytest.raises(ValueError, match="CUDA tensor"):
            pq.paged_attention(bad["q"], c.pages, bad["bt"], bad["seq_lens"], w.q_len, w.kv_dtype,
                               bad["ks"], bad["vs"], bad["out"])
        with pytest.raises(ValueError, match="CUDA tensor"):
            pq.paged_attention_noalloc(bad["q"], c.pages, bad["bt"], bad["seq_lens"], w.q_len,
                                       w.kv_dtype, bad["ks"], bad["vs"], bad["out"])
    with pytest.raises(ValueError, match="CUDA tensor"):
        pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                           status=torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                           workspace=torch.zeros(1 << 20, dtype=torch.uint8))
    k = torch.zeros((4, w.num_kv_heads, 128), dtype=torch.float16, device="cuda")
    slots = torch.arange(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pq.kv_append_quant(k, k, slots, w.kv_dtype, c.ks, c.vs, c.pages)
    o = torch.zeros((2, 3, 128), dtype=torch.float32, device="cuda")
    lse = torch.zeros((2, 3), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pq.lse_merge(o, lse, torch.empty((3, 128), dtype=torch.float16, device="cuda"))
    # nothing was launched with a bad pointer: the pool still gives the oracle's answer
    assert_close(pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks,
                                    c.vs, out), c.oracle_attention(), "after the rejected calls")


def test_maximum_sequence_count():
    # 2048 sequences, the largest batch (the per-sequence tables fill most of
    # the shared memory): eight copies of a 256-sequence workload (the seeded
    # generator numbers at most 256 sequences), each copy in pages of its own
    pq = require_gpu()
    rng = np.random.default_rng(12)
    base = W.Workload("max_seqs", 81, rng.integers(5, 61, size=256).tolist(), 32, 8, 5,
                      W.FP8_E4M3, pool_slack=0.05)
    cb = Case(base)
    ref = cb.oracle_attention()
    big = W.Workload("max_seqs_x8", 81, base.seq_lens * 8, 32, 8, 5, W.FP8_E4M3, pool_slack=0.05)
    plan = W.plan_pool(big)
    pages = pq.new_pages(plan.num_pages, 8, W.FP8_E4M3, "cuda", fill=0)
    for s2 in range(big.num_seqs):
        L = big.seq_lens[s2]
        k, v = W.kv_tokens(base, s2 % 256, 0, L, "cuda")
        pq.kv_append_quant(k, v, torch.from_numpy(W.slots_for(plan, s2, 0, L)).cuda(),
                           W.FP8_E4M3, cb.ks, cb.vs, pages)
    q = cb.q.repeat(8, 1, 1).contiguous()
    bt = torch.from_numpy(plan.block_table).cuda()
    sl = torch.tensor(big.seq_lens, dtype=torch.int32, device="cuda")
    for ns in (0, 7):
        out = torch.empty_like(q)
        pq.paged_attention(q, pages, bt, sl, 5, W.FP8_E4M3, cb.ks, cb.vs, out, num_splits=ns)
        o = out.float().cpu().numpy().reshape(8, 256 * 5, 32, 128)
        for copy in range(8):
            assert_close(o[copy], ref, "2048 sequences copy %d splits=%d" % (copy, ns))


@pytest.mark.parametrize("L", [1, 7, 16, 100, 513, 1024])
@pytest.mark.parametrize("hint", ["none", "exact"])
def test_one_segment_fp16_decode_with_empty_shares(L, hint):
    """One sequence on one kv-head, FP16, 8 query rows: a split over up to 8
    blocks is launched as a thread-block cluster whose blocks merge in shared
    memory.  The block table has room for 1024 tokens, so without a length
    hint the grid is sized for 1024 and, for short sequences, some blocks
    (block 0 too, for L = 1) get empty shares; they must still take part in
    the merge."""
    w = W.Workload("one_segment", 90 + L, [L], 8, 1, 1, W.FP16, outliers=False, pool_slack=0.5)
    c = Case(w)
    bt = torch.full((1, 64), -1, dtype=torch.int32, device="cuda")
    bt[:, :c.bt.shape[1]] = c.bt
    out = c.attention(bt=bt, max_seq_len=(L if hint == "exact" else 0))
    assert_close(out, c.oracle_attention(), "L %d hint %s" % (L, hint))
