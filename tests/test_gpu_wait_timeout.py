"""Failure detection without a GPU fault: every wait in the attention kernel is
bounded, and a wait that runs out ends in an error status the host reads, not
in a hang.

The testing entry point runs the E4M3 verify kernel with one page's tile copy
never issued (an mbarrier that nothing completes) and a 1 ms wait limit.  The
kernel must return, report PQKV_DEV_TIMEOUT, leave no copy in flight (the
context stays usable), and a normal call afterwards -- with the workspace
zeroed again, as the header requires after a timeout -- must match the
oracle.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import Case, assert_close, require_gpu

pytestmark = pytest.mark.gpu

DEV_TIMEOUT = 8


def _testing_entry(pq):
    lib = pq.load_library()
    fn = lib.pqkv_testing_attention_wait_timeout
    c_i32, c_i64, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    fn.restype = ctypes.c_int
    fn.argtypes = [c_vp, c_vp, c_vp, c_i64, c_vp, c_i32, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32,
                   c_i32, c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_sz, c_vp, c_vp, c_i32,
                   c_i32]
    return fn


def _run_test_mode(pq, c, out, ws, status, num_splits, skip_block, skip_page):
    w = c.w
    fn = _testing_entry(pq)
    p = ctypes.c_void_p
    return fn(p(c.q.data_ptr()), p(out.data_ptr()), p(c.pages.data_ptr()), c.pages.shape[0],
              p(c.bt.data_ptr()), c.bt.shape[1], p(c.seq_lens.data_ptr()), w.num_seqs, w.q_len,
              w.num_q_heads, w.num_kv_heads, 128, 16, w.kv_dtype, p(c.ks.data_ptr()),
              p(c.vs.data_ptr()), 0, num_splits, max(w.seq_lens), p(ws.data_ptr()),
              ws.numel(), p(status.data_ptr()), p(torch.cuda.current_stream().cuda_stream),
              skip_block, skip_page)


@pytest.mark.parametrize("num_splits,skip_block,skip_page", [(0, 0, 3), (0, 97, 0), (3, 5, 10)])
def test_a_wait_that_runs_out_reports_timeout_and_returns(num_splits, skip_block, skip_page):
    pq = require_gpu()
    w = W.workload("e4m3_verify_512k_stress", scale=0.004)
    c = Case(w, with_oracle=True)
    ws = torch.zeros(pq.workspace_size(w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads,
                                       num_splits), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(c.q, float("nan"))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _run_test_mode(pq, c, out, ws, status, num_splits, skip_block, skip_page) == 0
    torch.cuda.synchronize()               # returns: no hang, no CUDA error
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & DEV_TIMEOUT, "the wait that ran out was not reported"
    assert elapsed < 5.0
    assert "pipeline wait timed out" in pq.status_bits(status)

    # the context is still usable: a normal call after re-zeroing the workspace
    ws.zero_()
    status.zero_()
    out2 = torch.empty_like(c.q)
    pq.paged_attention(c.q, c.pages, c.bt, c.seq_lens, w.q_len, w.kv_dtype, c.ks, c.vs, out2,
                       num_splits=num_splits, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out2, c.oracle_attention(), "after a timeout")


def test_test_mode_without_a_skipped_copy_is_the_normal_kernel():
    """A skip position past the block's share skips nothing: no timeout, and
    the output matches the oracle."""
    pq = require_gpu()
    w = W.workload("e4m3_verify_512k_stress", scale=0.004)
    c = Case(w, with_oracle=True)
    ws = torch.zeros(pq.workspace_size(w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads, 0),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(c.q)
    assert _run_test_mode(pq, c, out, ws, status, 0, 0, 1 << 30) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, c.oracle_attention(), "test mode, nothing skipped")


def test_testing_entry_rejects_other_shapes():
    pq = require_gpu()
    w = W.workload("int8_decode_append_262k", scale=0.004)
    c = Case(w, with_oracle=False)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(c.q)
    assert _run_test_mode(pq, c, out, ws, status, 0, 0, 0) == -2     # PQKV_EUNSUPPORTED
