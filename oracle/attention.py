"""Oracle: quantize-and-append into a paged pool, paged decode / verify
attention, and split-KV partials merged by log-sum-exp.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg use it.

Everything here is plain float64 numpy in the order the definitions give it.

Pool layout (a choice of this library; the pages fix none): the pool is an
array [num_pages, Hkv, 2, page_size, D] -- for every page and kv-head a K tile
of page_size rows followed by a V tile -- of 1-byte codes (E4M3, INT8) or fp16
bit patterns (FP16).  Slot t of the pool is token t % page_size of page
t // page_size.  The ReVolta v0.1.3 release note ("Known issues") fixes
16-token kernel pages.

Attention (ReVolta README, "Quick start": MTP verify with 4 speculative
tokens; "Weight and KV formats": KV stored compressed and widened for compute):
for sequence s with L cached tokens (the q_len new ones included), query row i
of q_len sits at position p_i = L - q_len + i and attends to tokens j <= p_i.
Query head hq reads kv-head hq // (Hq / Hkv).  Scores are q . K_j / sqrt(D)
with K_j = dec(kcode_j) * k_scale; the output is sum_j softmax_j V_j.

Split-KV (the single-GPU counterpart of the decode-context-parallel split on
the ReVolta README, "Hardware" / "Quick start": TP4 + DCP2): each partition p
of the key range yields (O_p, m_p, l_p) with m_p the largest score, l_p the
sum of exp(score - m_p) and O_p the sum of exp(score - m_p) V_j; the result is
sum_p e^(m_p - M) O_p / sum_p e^(m_p - M) l_p with M = max_p m_p.
"""
from __future__ import annotations

import numpy as np

from .codec import INT8_TOKEN, dequantize, int8_row_scale, quantize


def new_pool(num_pages, num_kv_heads, head_dim, kv_dtype, page_size=16, fill=0):
    dt = np.uint16 if kv_dtype == 0 else np.uint8
    return np.full((num_pages, num_kv_heads, 2, page_size, head_dim), fill, dtype=dt)


def new_scale_pool(num_pages, num_kv_heads, page_size=16):
    """Per-row scales of a format-3 pool: float32 [num_pages, Hkv, page_size]
    (one for K and one for V), slot t of the pool at [t // P, :, t % P]."""
    return np.zeros((num_pages, num_kv_heads, page_size), dtype=np.float32)


def kv_append_quant(k, v, slot_mapping, kv_dtype, k_scale, v_scale, pages):
    """Return a copy of ``pages`` with the codes of k and v written at their slots.

    k, v: fp16 [T, Hkv, D]; slot_mapping: int [T] (negative = skip the token);
    k_scale, v_scale: one value, or one per kv-head.  Tokens are written in
    order, so a later token wins if two share a slot.

    Format 3 (INT8 with a scale per row): k_scale and v_scale are the scale
    pools [num_pages, Hkv, P]; every written row's scale is computed from the
    row and stored at its slot, and (pages, k_scale, v_scale) copies are
    returned.
    """
    if kv_dtype == INT8_TOKEN:
        return _append_row_scaled(k, v, slot_mapping, k_scale, v_scale, pages)
    k = np.asarray(k, dtype=np.float16)
    v = np.asarray(v, dtype=np.float16)
    out = np.array(pages, copy=True)
    P = out.shape[3]
    H = k.shape[1]
    ks = np.broadcast_to(np.asarray(k_scale, dtype=np.float32).reshape(-1), (H,))
    vs = np.broadcast_to(np.asarray(v_scale, dtype=np.float32).reshape(-1), (H,))
    slots = np.asarray(slot_mapping, dtype=np.int64).reshape(-1)
    keep = np.nonzero(slots >= 0)[0]
    if keep.size == 0:
        return out
    if slots[keep].max() >= out.shape[0] * P:
        raise IndexError("slot %d outside the pool" % slots[keep].max())
    # a later token wins: keep only the last occurrence of each slot
    _, last_rev = np.unique(slots[keep][::-1], return_index=True)
    keep = np.sort(keep[::-1][last_rev])
    page, off = np.divmod(slots[keep], P)
    for h in range(H):
        out[page, h, 0, off] = quantize(k[keep, h], ks[h], kv_dtype)
        out[page, h, 1, off] = quantize(v[keep, h], vs[h], kv_dtype)
    return out


def _append_row_scaled(k, v, slot_mapping, k_pool, v_pool, pages):
    k = np.asarray(k, dtype=np.float16)
    v = np.asarray(v, dtype=np.float16)
    out = np.array(pages, copy=True)
    kp = np.array(k_pool, dtype=np.float32, copy=True)
    vp = np.array(v_pool, dtype=np.float32, copy=True)
    P = out.shape[3]
    slots = np.asarray(slot_mapping, dtype=np.int64).reshape(-1)
    keep = np.nonzero(slots >= 0)[0]
    if keep.size == 0:
        return out, kp, vp
    if slots[keep].max() >= out.shape[0] * P:
        raise IndexError("slot %d outside the pool" % slots[keep].max())
    _, last_rev = np.unique(slots[keep][::-1], return_index=True)
    keep = np.sort(keep[::-1][last_rev])
    page, off = np.divmod(slots[keep], P)
    for h in range(k.shape[1]):
        ks = int8_row_scale(k[keep, h])
        vs = int8_row_scale(v[keep, h])
        out[page, h, 0, off] = quantize(k[keep, h], ks, INT8_TOKEN)
        out[page, h, 1, off] = quantize(v[keep, h], vs, INT8_TOKEN)
        kp[page, h, off] = ks
        vp[page, h, off] = vs
    return out, kp, vp


def gather_kv(pages, block_row, L, h, kv_dtype, k_scale, v_scale):
    """Dequantized float64 K and V [L, D] of one sequence and kv-head, read
    page by page through its block-table row.  For format 3 the scales are the
    scale pools and each row takes the scale stored at its slot."""
    P = pages.shape[3]
    n = (L + P - 1) // P
    ids = np.asarray(block_row[:n], dtype=np.int64)
    kc = pages[ids, h, 0].reshape(n * P, -1)[:L]
    vc = pages[ids, h, 1].reshape(n * P, -1)[:L]
    if kv_dtype == INT8_TOKEN:
        k_scale = np.asarray(k_scale)[ids, h].reshape(-1)[:L]
        v_scale = np.asarray(v_scale)[ids, h].reshape(-1)[:L]
    return dequantize(kc, k_scale, kv_dtype), dequantize(vc, v_scale, kv_dtype)


def _scale_of(scale, h):
    a = np.asarray(scale, dtype=np.float32).reshape(-1)
    return a[h] if a.size > 1 else a[0]


def attention_partial(qrows, K, V, limits, j0, j1, lower=None):
    """Partial softmax state of query rows over keys [j0, j1).

    qrows: float64 [R, D]; K, V: float64 [L, D]; limits[r]: last key position
    row r may see; lower[r] (optional): first key position row r may see.
    Returns (O [R, D], m [R], l [R]) with natural-log scores; rows that see no
    key of the range get m = -inf, l = 0, O = 0.
    """
    D = qrows.shape[1]
    R = qrows.shape[0]
    O = np.zeros((R, D))
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    if j1 <= j0:
        return O, m, l
    S = (qrows @ K[j0:j1].T) / np.sqrt(D)
    pos = np.arange(j0, j1)
    visible = pos[None, :] <= np.asarray(limits)[:, None]
    if lower is not None:
        visible &= pos[None, :] >= np.asarray(lower)[:, None]
    S = np.where(visible, S, -np.inf)
    for r in range(R):
        if not visible[r].any():
            continue
        m[r] = S[r].max()
        p = np.exp(S[r] - m[r])
        l[r] = p.sum()
        O[r] = p @ V[j0:j1]
    return O, m, l


def lse_merge(parts):
    """Merge partial states [(O_p, m_p, l_p), ...] into normalized outputs."""
    ms = np.stack([p[1] for p in parts])            # [P, R]
    M = ms.max(axis=0)
    w = np.exp(ms - M[None, :])                     # e^(m_p - M); 0 for empty parts
    num = sum(w[i][:, None] * parts[i][0] for i in range(len(parts)))
    den = sum(w[i] * parts[i][2] for i in range(len(parts)))
    return num / den[:, None]


def _rows_of(q, s, h, q_len, G):
    """Query rows of (sequence s, kv-head h): row r = i * G + g is query i of
    q-head h * G + g.  Returns float64 [q_len * G, D]."""
    blk = np.asarray(q[s * q_len:(s + 1) * q_len, h * G:(h + 1) * G], dtype=np.float64)
    return blk.reshape(q_len * G, -1)


def paged_attention(q, pages, block_table, seq_lens, q_len, kv_dtype, k_scale, v_scale,
                    num_splits=1, seqs=None, heads=None, window=0):
    """float64 attention output [B * q_len, Hq, D] (rows of sequences / heads
    not selected by ``seqs`` / ``heads`` are left NaN).

    ``num_splits`` > 1 cuts every sequence's key range into that many
    near-equal partitions and merges them by log-sum-exp.  ``window`` > 0
    limits query position p to the ``window`` most recent keys, itself
    included: keys p - window + 1 .. p (ReVolta README, "DFlash2 speculative
    decoding": sliding-window layers with a 2048-token window).
    """
    q = np.asarray(q)
    BQ, Hq, D = q.shape
    H = pages.shape[1]
    G = Hq // H
    out = np.full((BQ, Hq, D), np.nan)
    B = len(seq_lens)
    for s in (range(B) if seqs is None else seqs):
        L = int(seq_lens[s])
        limits = np.repeat(L - q_len + np.arange(q_len), G)
        lower = limits - window + 1 if window > 0 else None
        for h in (range(H) if heads is None else heads):
            if kv_dtype == INT8_TOKEN:
                K, V = gather_kv(pages, block_table[s], L, h, kv_dtype, k_scale, v_scale)
            else:
                K, V = gather_kv(pages, block_table[s], L, h, kv_dtype,
                                 _scale_of(k_scale, h), _scale_of(v_scale, h))
            rows = _rows_of(q, s, h, q_len, G)
            bounds = [(L * p) // num_splits for p in range(num_splits + 1)]
            parts = [attention_partial(rows, K, V, limits, bounds[p], bounds[p + 1], lower)
                     for p in range(num_splits)]
            o = lse_merge(parts).reshape(q_len, G, D)
            out[s * q_len:(s + 1) * q_len, h * G:(h + 1) * G] = o
    return out


def paged_attention_partial(q, pages, block_table, seq_lens, q_pos, q_len, kv_dtype, k_scale,
                            v_scale):
    """One rank's share of a decode context parallel split: attention over the
    keys held locally (seq_lens[s] of them), query i of sequence s seeing local
    keys j <= q_pos[s] + i.  Returns float64 (O / l [B * q_len, Hq, D],
    lse [B * q_len, Hq]) with lse = m + ln l in natural-log units; a row that
    sees no key gets O = 0 and lse = -inf."""
    q = np.asarray(q)
    BQ, Hq, D = q.shape
    H = pages.shape[1]
    G = Hq // H
    o = np.zeros((BQ, Hq, D))
    lse = np.full((BQ, Hq), -np.inf)
    for s in range(len(seq_lens)):
        L = int(seq_lens[s])
        limits = np.repeat(int(q_pos[s]) + np.arange(q_len), G)
        for h in range(H):
            if L == 0:
                continue
            if kv_dtype == INT8_TOKEN:
                K, V = gather_kv(pages, block_table[s], L, h, kv_dtype, k_scale, v_scale)
            else:
                K, V = gather_kv(pages, block_table[s], L, h, kv_dtype,
                                 _scale_of(k_scale, h), _scale_of(v_scale, h))
            O, m, l = attention_partial(_rows_of(q, s, h, q_len, G), K, V, limits, 0, L)
            seen = l > 0
            O[seen] /= l[seen][:, None]
            lr = np.where(seen, m + np.log(np.where(seen, l, 1.0)), -np.inf)
            o[s * q_len:(s + 1) * q_len, h * G:(h + 1) * G] = O.reshape(q_len, G, D)
            lse[s * q_len:(s + 1) * q_len, h * G:(h + 1) * G] = lr.reshape(q_len, G)
    return o, lse


def merge_lse(parts_o, parts_lse):
    """Combine partial results in (O / l, lse) form over the leading axis:
    LSE = ln sum_p e^{lse_p}, O = sum_p e^{lse_p - LSE} O_p.  Rows with no
    finite lse_p give O = 0, LSE = -inf."""
    po = np.asarray(parts_o, dtype=np.float64)
    pl = np.asarray(parts_lse, dtype=np.float64)
    M = pl.max(axis=0)
    finite = np.isfinite(M)
    w = np.where(finite[None], np.exp(pl - np.where(finite, M, 0.0)[None]), 0.0)
    tot = w.sum(axis=0)
    o = np.einsum("p...,p...d->...d", w, po) / np.where(tot > 0, tot, 1.0)[..., None]
    lse = np.where(tot > 0, np.where(finite, M, 0.0) + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    return o, lse


def dense_attention(q_rows, K, V, limits):
    """Attention of query rows over dense float64 K, V [L, D] (no pages)."""
    O, m, l = attention_partial(np.asarray(q_rows, np.float64), K, V, limits, 0, K.shape[0])
    return O / l[:, None]
