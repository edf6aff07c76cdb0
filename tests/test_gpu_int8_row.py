"""INT8 with a scale per (token, kv-head) row, computed at append time (the
pages' own INT8 design), against the oracle: codes and row scales bit for bit,
attention within the usual bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, assert_close, require_gpu

pytestmark = pytest.mark.gpu
T3 = W.INT8_ROW


def _append_both(kvals, vvals, H, slots, num_pages, k_stride=None):
    pq = require_gpu()
    T = len(slots)
    k = torch.from_numpy(kvals.reshape(T, H, 128)).cuda()
    v = torch.from_numpy(vvals.reshape(T, H, 128)).cuda()
    if k_stride is not None:       # K as a column slice of a wider buffer
        big = torch.zeros((T, k_stride), dtype=torch.float16, device="cuda")
        big[:, 256:256 + H * 128] = k.reshape(T, -1)
        k = big[:, 256:256 + H * 128].view(T, H, 128)
    pages = pq.new_pages(num_pages, H, T3, "cuda", fill=0x5A)
    pq.row_scales(pages).fill_(float("nan"))          # unwritten rows keep NaN scales
    sl = torch.from_numpy(np.asarray(slots, dtype=np.int64)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pq.kv_append_quant(k, v, sl, T3, None, None, pages, status=status)
    got_codes = pages.cpu().numpy()
    got_scales = pq.row_scales(pages).reshape(num_pages, H, 2, 16).cpu().numpy()
    pool = oracle.new_pool(num_pages, H, 128, T3, fill=0x5A)
    kp = np.full((num_pages, H, 16), np.nan, np.float32)
    vp = np.full((num_pages, H, 16), np.nan, np.float32)
    ref_codes, kp, vp = oracle.kv_append_quant(kvals.reshape(T, H, 128), vvals.reshape(T, H, 128),
                                               slots, T3, kp, vp, pool)
    assert int(status.item()) == 0
    return got_codes, got_scales, ref_codes, kp, vp


def _fp16_bits(ref):
    """binary16 bits of the oracle's float32 scales, which hold binary16 values"""
    h = ref.astype(np.float16)
    ok = ~np.isnan(ref)
    assert np.array_equal(h[ok].astype(np.float32), ref[ok])
    return h.view(np.uint16)


def _same_scales(got, kp, vp):
    # bit-identical, NaN where nothing was written
    assert got.dtype == np.float16
    for gi, ref in ((0, kp), (1, vp)):
        a = got[:, :, gi].view(np.uint16)
        assert np.array_equal(np.isnan(got[:, :, gi]), np.isnan(ref))
        ok = ~np.isnan(ref)
        assert np.array_equal(a[ok], _fp16_bits(ref)[ok])


def test_every_fp16_value_in_rows_bit_exact():
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    x = x[np.isfinite(x)]
    x = np.concatenate([x, np.zeros((-len(x)) % 128, np.float16)])
    T = len(x) // 128
    rng = np.random.default_rng(3)
    slots = rng.permutation(T + 40)[:T]
    got_c, got_s, ref_c, kp, vp = _append_both(x, x[::-1].copy(), 1, slots, (T + 40) // 16 + 1)
    assert np.array_equal(got_c, ref_c)
    _same_scales(got_s, kp, vp)


def test_edge_rows_and_strided_input():
    # zero rows, NaN and +-Inf elements, subnormal-only rows, a lone huge value
    H, T = 2, 40
    rng = np.random.default_rng(4)
    k = rng.normal(0, 2, (T, H, 128)).astype(np.float16)
    v = rng.normal(0, 2, (T, H, 128)).astype(np.float16)
    k[0] = 0
    k[1, 0, 7] = np.nan
    k[2, 1, 9] = np.inf
    k[3, 0, :] = np.float16(2.0 ** -20) * np.sign(rng.normal(size=128)).astype(np.float16)
    k[4, 1, 100] = np.float16(60000.0)
    v[5, :, :] = -0.0
    v[6, 0, ::2] = np.nan
    slots = rng.permutation(T + 8)[:T]
    got_c, got_s, ref_c, kp, vp = _append_both(k, v, H, slots, (T + 8) // 16 + 1, k_stride=1024)
    assert np.array_equal(got_c, ref_c)
    _same_scales(got_s, kp, vp)


SMALL = {"int8_row_decode_262k": 0.004, "int8_row_verify_131k": 0.01}
_cases = {}


def case(name):
    if name not in _cases:
        _cases[name] = Case(W.workload(name, scale=SMALL[name]))
    return _cases[name]


@pytest.mark.parametrize("name", W.ROW_SCALED_NAMES)
def test_workload_pools_and_scales_bit_exact(name):
    pq = require_gpu()
    c = case(name)
    assert np.array_equal(c.gpu_pool_bytes(), c.pool_o)
    n, H = c.pages.shape[:2]
    got = pq.row_scales(c.pages).reshape(n, H, 2, 16).cpu().numpy()
    written = c.oracle_ks != 0                       # the oracle's pool starts at 0 like new_pages
    assert np.array_equal(got[:, :, 0].view(np.uint16), _fp16_bits(c.oracle_ks))
    assert np.array_equal(got[:, :, 1].view(np.uint16), _fp16_bits(c.oracle_vs))
    assert written.any()


@pytest.mark.parametrize("name", W.ROW_SCALED_NAMES)
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_attention_matches_oracle(name, num_splits):
    c = case(name)
    assert_close(c.attention(num_splits=num_splits), c.oracle_attention(),
                 "%s splits=%d" % (name, num_splits))


def test_stale_nan_scales_and_codes_past_the_end_are_ignored():
    pq = require_gpu()
    w = W.Workload("row_nan_tail", 79, [37, 50], 8, 2, 5, T3, pool_slack=0.5)
    c = Case(w, with_oracle=False)
    pool = pq.new_pages(c.plan.num_pages, 2, T3, "cuda", fill=0x80)
    pq.row_scales(pool).fill_(float("nan"))
    for s, L in enumerate(w.seq_lens):
        k, v = W.kv_tokens(w, s, 0, L, "cuda")
        pq.kv_append_quant(k, v, torch.from_numpy(W.slots_for(c.plan, s, 0, L)).cuda(), T3,
                           None, None, pool)
    c.pages = pool
    c.build_oracle(fill=0x80)
    out = c.attention(num_splits=0)
    assert torch.isfinite(out.float()).all()
    assert_close(out, c.oracle_attention(), "row-scaled NaN tail")


def test_out_of_range_page_id_reads_zeros_and_reports():
    pq = require_gpu()
    w = W.Workload("row_badpage", 80, [40], 4, 1, 1, T3, pool_slack=0.5)
    c = Case(w)
    bt = c.bt.clone()
    bt[0, 1] = 10 ** 6
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(c.q)
    pq.paged_attention(c.q, c.pages, bt, c.seq_lens, 1, T3, None, None, out, status=status)
    assert "block-table page id out of range" in pq.status_bits(status)
    spare = c.pool_o.shape[0]
    pool = np.concatenate([c.pool_o, np.zeros_like(c.pool_o[:1])])
    kp = np.concatenate([c.oracle_ks, np.zeros_like(c.oracle_ks[:1])])
    vp = np.concatenate([c.oracle_vs, np.zeros_like(c.oracle_vs[:1])])
    bt_np = c.plan.block_table.copy()
    bt_np[0, 1] = spare
    ref = oracle.paged_attention(c.q.cpu().numpy(), pool, bt_np, w.seq_lens, 1, T3, kp, vp)
    assert_close(out, ref, "row-scaled zero page")
