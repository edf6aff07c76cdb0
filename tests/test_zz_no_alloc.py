"""pqkv_paged_attention_noalloc: attention for callers that cannot allocate
device memory (for example a runtime that budgets all GPU memory up front and
forbids cudaMalloc at call time).  It must give the same result as
pqkv_paged_attention with a caller workspace, call after call, although its
scratch area keeps the previous call's contents.

Kept in a file of its own that is collected after every other test file.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import Case, assert_close, require_gpu

pytestmark = pytest.mark.gpu


def _noalloc(pq, c, out, num_splits=0):
    w = c.w
    return pq.paged_attention_noalloc(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks,
                                      c.vs, out, num_splits=num_splits)


@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_workspace_entry_point_twice(num_splits):
    pq = require_gpu()
    c = Case(W.workload("e4m3_verify_512k_stress", scale=0.004), with_oracle=False)
    ref = c.attention(num_splits=num_splits)          # existing entry point, caller workspace
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    for call in range(2):                            # the scratch keeps the last call's contents
        out = torch.full_like(c.q, float("nan"))
        _noalloc(pq, c, out, num_splits)
        torch.cuda.synchronize()
        assert_close(out, ref64, "noalloc call %d splits %d" % (call, num_splits))


def test_noalloc_int8_decode_and_no_split():
    pq = require_gpu()
    c = Case(W.workload("int8_decode_append_262k", scale=0.004), with_oracle=False)
    for ns in (0, 1):
        ref = c.attention(num_splits=ns).float().cpu().numpy().astype(np.float64)
        out = torch.empty_like(c.q)
        _noalloc(pq, c, out, ns)
        assert_close(out, ref, "noalloc int8 splits %d" % ns)


def test_noalloc_row_scaled_int8_verify():
    pq = require_gpu()
    c = Case(W.workload("int8_row_verify_131k", scale=0.01), with_oracle=False)
    ref = c.attention(num_splits=0).float().cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full_like(c.q, float("nan"))
        _noalloc(pq, c, out, 0)
        torch.cuda.synchronize()
        assert_close(out, ref, "noalloc int8_row call %d" % call)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    pq = require_gpu()
    # 2048 sequences x 8 kv-heads in the balanced split need more than 16 MiB
    B, H, q_len, Hq = 2048, 8, 5, 32
    assert pq.workspace_size(B, q_len, Hq, H) > pq.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B * q_len, Hq, 128), dtype=torch.float16, device="cuda")
    pages = pq.new_pages(4, H, W.FP8_E4M3, "cuda", fill=0)
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    sl = torch.full((B,), 5, dtype=torch.int32, device="cuda")
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        pq.paged_attention_noalloc(q, pages, bt, sl, q_len, W.FP8_E4M3, one, one, torch.empty_like(q))


def test_noalloc_32_row_verify_against_the_oracle():
    """q_len 8 with 4 query heads per kv-head: 32 rows, the widest row tile.
    The scratch it needs is sized from the grid the call launches, so the
    default balanced split fits whatever the context length."""
    pq = require_gpu()
    c = Case(W.workload("e4m3_verify_q8_131k", scale=0.004), with_oracle=True)
    ref = c.oracle_attention()
    for call in range(2):
        out = torch.full_like(c.q, float("nan"))
        _noalloc(pq, c, out, 0)
        torch.cuda.synchronize()
        assert_close(out, ref, "noalloc 32 rows call %d" % call)


def test_noalloc_largest_fixed_split_that_fits():
    """The stress verify (8 sequences x 8 kv-heads, 24 padded rows) cut into
    21 fixed partitions per (sequence, kv-head) needs 16,773,376 bytes of
    scratch, just under the 16 MiB area; two calls in a row must both match
    the oracle (the merge counters are cleared between calls).  22 partitions
    no longer fit and are refused before anything is queued."""
    pq = require_gpu()
    c = Case(W.workload("e4m3_verify_512k_stress", scale=0.004), with_oracle=True)
    assert pq.workspace_size(8, 5, 32, 8, 21) == 16773376 <= pq.NOALLOC_SCRATCH_BYTES
    assert pq.workspace_size(8, 5, 32, 8, 22) > pq.NOALLOC_SCRATCH_BYTES
    ref = c.oracle_attention()
    for call in range(2):
        out = torch.full_like(c.q, float("nan"))
        _noalloc(pq, c, out, 21)
        torch.cuda.synchronize()
        assert_close(out, ref, "noalloc 21 splits call %d" % call)
    before = out.clone()
    with pytest.raises(ValueError):
        _noalloc(pq, c, out, 22)
    torch.cuda.synchronize()
    assert torch.equal(out, before)
    # a valid call after the refused one is still right
    out2 = torch.empty_like(c.q)
    _noalloc(pq, c, out2, 21)
    assert_close(out2, ref, "noalloc after a refused call")
