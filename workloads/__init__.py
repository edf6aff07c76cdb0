"""Seeded synthetic inputs for the paged quantized-KV path.

This module only *draws* inputs: fp16 query/key/value values, context lengths,
shuffled block tables, slot mappings and the per-layer scales that a calibration
would have produced (amax / 448 for E4M3, amax / 127 for INT8).  It contains
none of the arithmetic of the method itself (no encoding, no attention), so the
oracle and the CUDA path can both take their inputs from here without sharing
any of the computation that is being checked.

Value generator
---------------
Every fp16 value is a pure function of (seed, kind, sequence, kv-head, token,
dim).  A 42-bit counter is hashed with a 32-bit integer mixer (Chris Wellons'
"lowbias32" construction) written with exact int64 tensor arithmetic, so the
same bits come out on the CPU and on the GPU.  The top 16 hash bits index a
table of N(0,1) quantiles rounded to fp16; the low 16 bits mark about 1% of
elements as outliers, which are multiplied by 20 (in fp32, then rounded to
fp16).  Because it is counter-based, any slice (one sequence, one head, one
token range) can be regenerated on its own, which is what lets the oracle
check sampled outputs of multi-gigabyte workloads.

Workload shapes follow the serving setup on the ReVolta README ("Quick start",
launch: 8 concurrent sequences, 8192-token batch budget, 512K context through
YaRN, MTP4 verify with 4 speculative tokens, 16-token kernel pages from the
v0.1.3 release note, "Known issues").
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

M32 = (1 << 32) - 1

KIND_K = 0
KIND_V = 1
KIND_Q = 2
KIND_APPEND_K = 3
KIND_APPEND_V = 4

PAGE_SIZE = 16
HEAD_DIM = 128

# kv dtype names used throughout (the integer values match the C-ABI enum)
FP16 = 0
FP8_E4M3 = 1
INT8 = 2
INT8_ROW = 3          # INT8 with a scale per (token, kv-head) row, computed at append time
DTYPE_NAMES = {FP16: "fp16", FP8_E4M3: "fp8_e4m3", INT8: "int8"}

_TABLE_CACHE = {}


def normal_table() -> np.ndarray:
    """65,536 N(0,1) quantiles at the cell midpoints, rounded to fp16."""
    if "t" not in _TABLE_CACHE:
        from scipy.special import ndtri

        u = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
        _TABLE_CACHE["t"] = ndtri(u).astype(np.float16)
    return _TABLE_CACHE["t"]


def _mulmod32(x: torch.Tensor, c: int) -> torch.Tensor:
    # (x * c) mod 2**32 for 0 <= x < 2**32 without int64 overflow
    lo = x * (c & 0xFFFF)
    hi = ((x * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mulmod32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mulmod32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def hash32(counter: torch.Tensor, seed: int) -> torch.Tensor:
    """32-bit hash of a non-negative int64 counter (< 2**62) and a seed."""
    lo = counter & M32
    hi = counter >> 32
    s = _mix32(torch.full_like(hi, seed & M32) ^ hi)
    return _mix32(lo ^ s)


def _counter(kind, s, h, t, d):
    # kind < 8, s < 256, h < 64, t < 2**20, d < 128 -> 45 bits
    return ((((kind * 256 + s) * 64 + h) << 20) + t) * 128 + d


def draw_values(seed: int, kind: int, s: int, t0: int, t1: int, heads: Sequence[int] | int,
                dim: int, outliers: bool, device="cpu") -> torch.Tensor:
    """fp16 tensor [t1 - t0, len(heads), dim] of seeded N(0,1) values.

    With ``outliers`` about 1% of elements are multiplied by 20.
    """
    if isinstance(heads, int):
        heads = list(range(heads))
    assert dim <= HEAD_DIM and 0 <= t0 <= t1 <= (1 << 20) and s < 256
    table = torch.from_numpy(normal_table()).to(device)
    t = torch.arange(t0, t1, dtype=torch.int64, device=device).view(-1, 1, 1)
    hh = torch.tensor(list(heads), dtype=torch.int64, device=device).view(1, -1, 1)
    d = torch.arange(dim, dtype=torch.int64, device=device).view(1, 1, -1)
    hsh = hash32(_counter(kind, s, hh, t, d), seed)
    val = table[(hsh >> 16).long()]
    if outliers:
        mark = (hsh & 0xFFFF) < 655
        val = torch.where(mark, (val.float() * 20.0).half(), val)
    return val


def draw_values_chunked(seed, kind, s, t0, t1, heads, dim, outliers, device, chunk=1 << 16):
    out = []
    for a in range(t0, t1, chunk):
        out.append(draw_values(seed, kind, s, a, min(t1, a + chunk), heads, dim, outliers, device))
    if not out:
        nh = heads if isinstance(heads, int) else len(heads)
        return torch.empty((0, nh, dim), dtype=torch.float16, device=device)
    return torch.cat(out, 0)


def scale_from_amax(amax: float, qmax: float) -> float:
    """fp32(amax / qmax), correctly rounded (float64 division, one fp32 rounding)."""
    return float(np.float32(float(amax) / qmax))


# --------------------------------------------------------------------------
# Workload configurations
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    seq_lens: List[int]
    num_q_heads: int
    num_kv_heads: int
    q_len: int
    kv_dtype: int
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    outliers: bool = True
    scale_per_head: bool = False
    pool_slack: float = 0.0      # extra free pages in the pool, as a fraction
    append_tokens: int = 0       # size of an extra append chunk (fragmented pool)
    append_offset: int = 0       # chunk starts at this offset inside a page
    append_per_step: int = 0     # tokens appended per sequence per step
    max_splits: int = 64

    @property
    def num_seqs(self):
        return len(self.seq_lens)

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def rows(self):
        return self.group * self.q_len

    def pages_of(self, L):
        return (L + self.page_size - 1) // self.page_size

    @property
    def elem_bytes(self):
        return 2 if self.kv_dtype == FP16 else 1

    @property
    def row_scale_bytes(self):
        """bytes of stored scale per (token, kv-head): an fp16 K and V row
        scale for INT8_ROW, nothing for the other formats"""
        return 4 if self.kv_dtype == INT8_ROW else 0

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one attention pass must read: K and V of every
        cached token of every sequence and kv-head (with their row scales)."""
        rows = sum(self.seq_lens) * self.num_kv_heads
        return rows * (self.head_dim * 2 * self.elem_bytes + self.row_scale_bytes)

    def append_bytes(self, tokens: int) -> int:
        """Algorithmic bytes of one append of ``tokens`` tokens: fp16 K and V
        read, codes (and row scales) written, int64 slots read."""
        n = tokens * self.num_kv_heads * self.head_dim * 2
        return (n * 2 + n * self.elem_bytes + tokens * self.num_kv_heads * self.row_scale_bytes
                + tokens * 8)


def workload(name: str, scale: float = 1.0) -> Workload:
    """The five synthetic workloads.  ``scale`` < 1 shrinks context lengths
    (keeping every other property) to sizes the oracle finishes in seconds."""
    def L(x):
        if scale >= 1.0:
            return int(x)
        return max(PAGE_SIZE + 5, int(x * scale) | 5)  # odd-ish: ragged last page

    if name == "tiny_fp16_decode":
        return Workload(name, 1, [1024], 8, 1, 1, FP16, outliers=False, pool_slack=1.0)
    if name == "e4m3_decode_b8":
        rng = np.random.default_rng(np.random.SeedSequence([2, 0]))
        lens = rng.integers(2048, 32768, size=8, endpoint=True).tolist()
        return Workload(name, 2, [L(x) for x in lens], 32, 8, 1, FP8_E4M3, pool_slack=0.05)
    if name == "e4m3_verify_131k":
        return Workload(name, 3, [L(131072)] * 8, 32, 8, 5, FP8_E4M3, pool_slack=0.01)
    if name == "int8_decode_append_262k":
        return Workload(name, 4, [L(262144)] * 4, 32, 8, 1, INT8, scale_per_head=True,
                        pool_slack=0.01, append_per_step=1)
    if name == "int8_row_decode_262k":       # the 262K INT8 decode's shapes, run-time row scales
        return Workload(name, 6, [L(262144)] * 4, 32, 8, 1, INT8_ROW, pool_slack=0.01)
    if name == "int8_row_verify_131k":       # the 131K E4M3 verify's shapes, run-time row scales
        return Workload(name, 7, [L(131072)] * 8, 32, 8, 5, INT8_ROW, pool_slack=0.01)
    if name == "e4m3_verify_q8_131k":        # the 131K verify with 7 drafts + 1: 32 rows
        return Workload(name, 8, [L(131072)] * 8, 32, 8, 8, FP8_E4M3, pool_slack=0.01)
    if name == "e4m3_verify_512k_stress":
        return Workload(name, 5, [L(524288)] * 2 + [L(32768)] * 6, 32, 8, 5, FP8_E4M3,
                        pool_slack=0.02, append_tokens=8192 if scale >= 1.0 else 520,
                        append_offset=7)
    raise KeyError(name)


WORKLOAD_NAMES = ["tiny_fp16_decode", "e4m3_decode_b8", "e4m3_verify_131k",
                  "int8_decode_append_262k", "e4m3_verify_512k_stress"]
# INT8 with run-time row scales (the README's own INT8 design) on the 262K decode's and
# the 131K verify's shapes
ROW_SCALED_NAMES = ["int8_row_decode_262k", "int8_row_verify_131k"]
# the wider verify: q_len 8 (a 7-token draft), 32 query rows per kv-head
WIDE_VERIFY_NAMES = ["e4m3_verify_q8_131k"]


@dataclasses.dataclass
class PoolPlan:
    num_pages: int
    max_pages_per_seq: int
    block_table: np.ndarray          # int32 [B, max_pages_per_seq], -1 padded
    append_slots: Optional[np.ndarray] = None   # int64 [append_tokens] (fragmented chunk)


def plan_pool(w: Workload, extra_tokens_per_seq: int = 0) -> PoolPlan:
    """Shuffled page assignment: every sequence gets its pages from a seeded
    permutation of the pool, so consecutive logical pages are scattered.

    ``extra_tokens_per_seq`` reserves room for tokens appended later.  When the
    workload has an append chunk, it goes into a disjoint, shuffled set of free
    pages and starts ``append_offset`` tokens into its first page.
    """
    rng = np.random.default_rng(np.random.SeedSequence([w.seed, 1]))
    need = [w.pages_of(L + extra_tokens_per_seq) for L in w.seq_lens]
    chunk_pages = 0
    if w.append_tokens:
        chunk_pages = w.pages_of(w.append_tokens + w.append_offset)
    used = sum(need) + chunk_pages
    num_pages = used + max(1, int(math.ceil(used * w.pool_slack)))
    perm = rng.permutation(num_pages).astype(np.int64)
    maxp = max(need)
    bt = np.full((w.num_seqs, maxp), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    slots = None
    if w.append_tokens:
        # the remaining pages are the free list; take a random subset of them
        free = perm[pos:]
        chunk = rng.choice(free, size=chunk_pages, replace=False)
        t = np.arange(w.append_tokens, dtype=np.int64) + w.append_offset
        slots = chunk[t // w.page_size] * w.page_size + t % w.page_size
    return PoolPlan(num_pages, maxp, bt, slots)


def slots_for(plan: PoolPlan, s: int, t0: int, t1: int, page_size: int = PAGE_SIZE) -> np.ndarray:
    """Cache slots of tokens [t0, t1) of sequence s under the block table."""
    t = np.arange(t0, t1, dtype=np.int64)
    return plan.block_table[s, t // page_size].astype(np.int64) * page_size + t % page_size


def query(w: Workload, device="cpu") -> torch.Tensor:
    """fp16 queries [B * q_len, Hq, D], N(0,1) without outliers."""
    parts = [draw_values(w.seed, KIND_Q, s, 0, w.q_len, w.num_q_heads, w.head_dim, False, device)
             for s in range(w.num_seqs)]
    return torch.cat(parts, 0).contiguous()


def kv_tokens(w: Workload, s: int, t0: int, t1: int, device="cpu", heads=None):
    """fp16 K and V [t1 - t0, Hkv, D] of tokens [t0, t1) of sequence s."""
    heads = w.num_kv_heads if heads is None else heads
    k = draw_values_chunked(w.seed, KIND_K, s, t0, t1, heads, w.head_dim, w.outliers, device)
    v = draw_values_chunked(w.seed, KIND_V, s, t0, t1, heads, w.head_dim, w.outliers, device)
    return k, v


def append_chunk(w: Workload, device="cpu"):
    """fp16 K and V of the extra append chunk [append_tokens, Hkv, D]."""
    k = draw_values_chunked(w.seed, KIND_APPEND_K, 0, 0, w.append_tokens, w.num_kv_heads,
                            w.head_dim, w.outliers, device)
    v = draw_values_chunked(w.seed, KIND_APPEND_V, 0, 0, w.append_tokens, w.num_kv_heads,
                            w.head_dim, w.outliers, device)
    return k, v


def step_tokens(w: Workload, plan: PoolPlan, device="cpu"):
    """The decode step's own append, ``append_per_step`` tokens per sequence:
    the newest tokens of every sequence (the ones its query sees last), as
    fp16 K and V [B * n, Hkv, D] with their slots int64 [B * n].  They are the
    values the pool already holds at those slots, so re-appending them every
    step is idempotent and a timed loop stays in steady state."""
    n = w.append_per_step
    ks, vs, sl = [], [], []
    for s, L in enumerate(w.seq_lens):
        k, v = kv_tokens(w, s, L - n, L, device)
        ks.append(k)
        vs.append(v)
        sl.append(slots_for(plan, s, L - n, L))
    return torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), np.concatenate(sl)


def step_append_tokens(w: Workload) -> int:
    """Tokens one timed step appends: the extra chunk, or the decode step's
    own tokens."""
    return w.append_tokens or w.num_seqs * w.append_per_step


def calibrated_scales(w: Workload, device="cpu"):
    """Per-layer (or per-kv-head for INT8) scales: amax of the layer's fp16 K
    (resp. V) over every cached token, divided by the format's largest value.

    Returns float32 tensors of shape [1] or [Hkv] on ``device``.  FP16 and
    INT8_ROW pools take no scale argument; ones are returned so callers can
    pass something.
    """
    H = w.num_kv_heads
    if w.kv_dtype in (FP16, INT8_ROW):
        one = torch.ones(H if w.scale_per_head else 1, dtype=torch.float32, device=device)
        return one, one.clone()
    qmax = 448.0 if w.kv_dtype == FP8_E4M3 else 127.0
    ka = torch.zeros(H, dtype=torch.float32, device=device)
    va = torch.zeros(H, dtype=torch.float32, device=device)
    for s, L in enumerate(w.seq_lens):
        for a in range(0, L, 1 << 16):
            k, v = kv_tokens(w, s, a, min(L, a + (1 << 16)), device)
            ka = torch.maximum(ka, k.float().abs().amax(dim=(0, 2)))
            va = torch.maximum(va, v.float().abs().amax(dim=(0, 2)))
    if w.scale_per_head:
        ks = [scale_from_amax(x, qmax) for x in ka.tolist()]
        vs = [scale_from_amax(x, qmax) for x in va.tolist()]
    else:
        ks = [scale_from_amax(ka.max().item(), qmax)]
        vs = [scale_from_amax(va.max().item(), qmax)]
    return (torch.tensor(ks, dtype=torch.float32, device=device),
            torch.tensor(vs, dtype=torch.float32, device=device))
