"""Sliding-window attention (pqkv_paged_attention_window) against the oracle:
query position p sees keys p - window + 1 .. p.  Covers the row widths of
every kernel shape (8 rows with one kv-head, 4 / 20 / 32 rows with eight),
the four KV formats, windows from one key to wider than the cache, both split
modes, and that pages lying wholly before every query's window are never read
(they are filled with NaN codes on the GPU only)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, assert_close, require_gpu

pytestmark = pytest.mark.gpu

# shapes beyond the workloads: 16 rows (q_len 4, four q-heads per kv-head) and an
# FP16 pool with 20 rows
EXTRA = {
    "rows16_e4m3": lambda: W.Workload("rows16_e4m3", 21, [300, 77, 1029], 32, 8, 4, W.FP8_E4M3,
                                      pool_slack=0.1),
    "rows20_fp16": lambda: W.Workload("rows20_fp16", 22, [200, 41], 32, 8, 5, W.FP16,
                                      outliers=False, pool_slack=0.1),
}

CASES = [
    ("e4m3_verify_512k_stress", 0.004, [1, 16, 17, 100, 1000]),   # 20 rows, E4M3
    ("e4m3_verify_q8_131k", 0.004, [7, 300]),                     # 32 rows
    ("int8_decode_append_262k", 0.004, [1, 64, 513]),             # 4 rows, INT8 per-head scales
    ("int8_row_verify_131k", 0.004, [33, 400]),                   # 20 rows, INT8 row scales
    ("tiny_fp16_decode", 1.0, [1, 2, 200, 1023, 1024]),           # 8 rows on one kv-head, FP16
    ("rows16_e4m3", None, [5, 64, 700]),
    ("rows20_fp16", None, [3, 50]),
]


def _oracle_window(c, window):
    w = c.w
    return oracle.paged_attention(c.q.cpu().numpy(), c.pool_o, c.plan.block_table, w.seq_lens,
                                  w.q_len, w.kv_dtype, c.oracle_ks, c.oracle_vs, window=window)


@pytest.mark.parametrize("name,scale,windows", CASES)
def test_window_matches_the_oracle(name, scale, windows):
    pq = require_gpu()
    c = Case(EXTRA[name]() if scale is None else W.workload(name, scale), with_oracle=True)
    w = c.w
    for window in windows:
        for ns in (0, 3):
            out = torch.full_like(c.q, float("nan"))
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs,
                               out, num_splits=ns, window=window, status=status,
                               max_seq_len=max(w.seq_lens))
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert_close(out, _oracle_window(c, window), "%s window %d splits %d" % (name, window, ns))


def test_window_wider_than_the_cache_is_plain_attention():
    pq = require_gpu()
    c = Case(W.workload("e4m3_verify_512k_stress", 0.004), with_oracle=False)
    ref = c.attention()
    w = c.w
    out = torch.empty_like(c.q)
    pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                       window=10 ** 6)
    assert_close(out, ref.float().cpu().numpy().astype(np.float64), "window > cache")
    out0 = torch.empty_like(c.q)
    pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out0,
                       window=0)
    assert torch.equal(out0, ref)                       # window 0 is the plain call


@pytest.mark.parametrize("name,scale,window", [("e4m3_verify_512k_stress", 0.004, 40),
                                               ("tiny_fp16_decode", 1.0, 100),
                                               ("int8_row_verify_131k", 0.004, 50)])
def test_pages_before_the_window_are_not_read(name, scale, window):
    """Pages whose tokens all precede every query's window get NaN codes (and
    NaN row scales) on the GPU; the output must stay finite and match the
    oracle on the clean pool."""
    pq = require_gpu()
    c = Case(W.workload(name, scale), with_oracle=True)
    w = c.w
    ref = _oracle_window(c, window)
    nan_code = {W.FP16: 0x7E00, W.FP8_E4M3: 0x7F, W.INT8: 0x80, W.INT8_ROW: 0x80}[w.kv_dtype]
    poisoned = 0
    for s, L in enumerate(w.seq_lens):
        first_key = max(0, L - w.q_len - window + 1)
        for pg in range(first_key // 16):                   # wholly before the window
            page = int(c.plan.block_table[s, pg])
            if w.kv_dtype == W.FP16:
                c.pages[page].view(torch.int16).fill_(nan_code)
            else:
                c.pages[page].fill_(nan_code)
                if w.kv_dtype == W.INT8_ROW:
                    pq.row_scales(c.pages)[page].fill_(float("nan"))
            poisoned += 1
    assert poisoned > 0
    out = torch.empty_like(c.q)
    pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out,
                       window=window)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert_close(out, ref, "%s window %d over poisoned pages" % (name, window))


def test_negative_window_is_rejected():
    pq = require_gpu()
    c = Case(W.workload("tiny_fp16_decode"), with_oracle=False)
    w = c.w
    with pytest.raises(ValueError):
        pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs,
                           torch.empty_like(c.q), window=-1)
