"""Shared set-up for the GPU parity tests: build the same paged pool on the GPU
(through the library's kv_append_quant) and in the oracle (through its own
encoder), from the seeded generator in ``workloads``."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W

ATOL = 2e-3
RTOL = 1e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    import paged_quantized_kv_append_gb300 as pq
    pq.load_library()   # raises if the CUDA library is missing: no fallback
    return pq


class Case:
    """A workload materialised on the GPU and (optionally) in the oracle."""

    def __init__(self, w: W.Workload, with_oracle=True, fill=0):
        pq = require_gpu()
        self.w = w
        self.plan = W.plan_pool(w)
        dev = "cuda"
        self.ks, self.vs = W.calibrated_scales(w, device=dev)
        self.pages = pq.new_pages(self.plan.num_pages, w.num_kv_heads, w.kv_dtype, dev, fill=fill)
        self.bt = torch.from_numpy(self.plan.block_table).to(dev)
        self.seq_lens = torch.tensor(w.seq_lens, dtype=torch.int32, device=dev)
        for s, L in enumerate(w.seq_lens):
            for a in range(0, L, 1 << 16):
                b = min(L, a + (1 << 16))
                k, v = W.kv_tokens(w, s, a, b, dev)
                slots = torch.from_numpy(W.slots_for(self.plan, s, a, b)).to(dev)
                pq.kv_append_quant(k, v, slots, w.kv_dtype, self.ks, self.vs, self.pages)
        self.q = W.query(w, dev)
        self.pool_o = None
        if with_oracle:
            self.build_oracle(fill)

    def build_oracle(self, fill=0):
        w = self.w
        pool = oracle.new_pool(self.plan.num_pages, w.num_kv_heads, w.head_dim, w.kv_dtype, fill=fill)
        if w.kv_dtype == W.INT8_ROW:
            ks = oracle.new_scale_pool(self.plan.num_pages, w.num_kv_heads)
            vs = oracle.new_scale_pool(self.plan.num_pages, w.num_kv_heads)
        else:
            ks, vs = self.ks.cpu().numpy(), self.vs.cpu().numpy()
        for s, L in enumerate(w.seq_lens):
            k, v = W.kv_tokens(w, s, 0, L, "cpu")
            r = oracle.kv_append_quant(k.numpy(), v.numpy(), W.slots_for(self.plan, s, 0, L),
                                       w.kv_dtype, ks, vs, pool)
            if w.kv_dtype == W.INT8_ROW:
                pool, ks, vs = r
            else:
                pool = r
        self.pool_o = pool
        self.oracle_ks, self.oracle_vs = ks, vs

    def gpu_pool_bytes(self):
        x = self.pages.cpu()
        return x.view(torch.int16).numpy().view(np.uint16) if self.w.kv_dtype == W.FP16 else x.numpy()

    def attention(self, num_splits=0, bt=None, out=None, max_seq_len=0):
        pq = require_gpu()
        out = torch.empty_like(self.q) if out is None else out
        pq.paged_attention(self.q, self.pages, self.bt if bt is None else bt, self.seq_lens,
                           self.w.q_len, self.w.kv_dtype, self.ks, self.vs, out,
                           num_splits=num_splits, max_seq_len=max_seq_len)
        return out

    def oracle_attention(self, seqs=None, heads=None):
        w = self.w
        return oracle.paged_attention(self.q.cpu().numpy(), self.pool_o, self.plan.block_table,
                                      w.seq_lens, w.q_len, w.kv_dtype, self.oracle_ks,
                                      self.oracle_vs, seqs=seqs, heads=heads)


def assert_close(gpu, ref, what=""):
    """|gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise, and a relative L2 bound."""
    g = gpu.float().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    sel = ~np.isnan(ref)
    g, r = g[sel].astype(np.float64), ref[sel]
    assert np.isfinite(g).all(), "%s: non-finite GPU output" % what
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    worst = np.argmax(err - bound)
    assert (err <= bound).all(), "%s: max excess %.3g at %d (gpu %.6g ref %.6g)" % (
        what, (err - bound)[worst], worst, g[worst], r[worst])
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert rel <= 1e-2, "%s: relative L2 error %.3g" % (what, rel)
    return float(err.max()), float(rel)
