"""Pins for the oracle's decode-context-parallel pieces: one rank's partial
attention over its share of the keys, and the log-sum-exp merge.

Pinned against a per-key brute-force loop (math.exp / math.log), scipy's
logsumexp, the already pinned full attention (a single share holding every
key must reproduce it), and the exact identity that merging any page-aligned
split of the keys gives the unsplit result.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from tests.test_oracle_attention import _random_case


def shares(bt, L, q_len, bounds):
    """Per-rank (block_table, seq_lens, q_pos) for page bounds [(p0, p1), ...]
    applied to every sequence (clamped to each sequence's pages)."""
    out = []
    for p0, p1 in bounds:
        B = len(L)
        lbt = np.zeros((B, max(1, p1 - p0)), dtype=np.int32)
        ls, qp = [], []
        for s in range(B):
            n = (L[s] + 15) // 16
            a, b = min(p0, n), min(p1, n)
            lbt[s, :b - a] = bt[s, a:b]
            ls.append(max(0, min(L[s], b * 16) - a * 16))
            qp.append(L[s] - q_len - a * 16)
        out.append((lbt, np.array(ls), np.array(qp)))
    return out


def test_single_share_is_full_attention_and_lse_matches_brute_force():
    rng = np.random.default_rng(21)
    L = [23, 40]
    q, pool, bt, L, ks, vs = _random_case(rng, L, 2, 2, 8, 5, 1)
    (lbt, ls, qp), = shares(bt, L, 5, [(0, 8)])
    o, lse = oracle.paged_attention_partial(q, pool, lbt, ls, qp, 5, 1, ks, vs)
    full = oracle.paged_attention(q, pool, bt, L, 5, 1, ks, vs)
    assert np.allclose(o, full, rtol=1e-13, atol=1e-14)
    # brute force: lse of row (s, i, hq) = ln sum_j exp(score_j) over visible keys
    D = q.shape[2]
    for s in range(len(L)):
        for i in range(5):
            for hq in range(q.shape[1]):
                h = hq // 2
                acc = []
                for j in range(L[s] - 5 + i + 1):
                    page = bt[s, j // 16]
                    kr = oracle.dequantize(pool[page, h, 0, j % 16], ks[0], 1)
                    acc.append(math.fsum(float(a) * float(b) for a, b in zip(q[s * 5 + i, hq], kr))
                               / math.sqrt(D))
                mx = max(acc)
                want = mx + math.log(math.fsum(math.exp(x - mx) for x in acc))
                assert abs(lse[s * 5 + i, hq] - want) < 1e-12


@pytest.mark.parametrize("bounds", [[(0, 1), (1, 8)], [(0, 2), (2, 3), (3, 8)],
                                    [(0, 3), (3, 8), (8, 9)]])   # the last share is empty
def test_merged_shares_equal_full_attention(bounds):
    rng = np.random.default_rng(22)
    q, pool, bt, L, ks, vs = _random_case(rng, [37, 50, 6], 2, 4, 16, 5, 2, scale_per_head=True)
    parts = [oracle.paged_attention_partial(q, pool, lbt, ls, qp, 5, 2, ks, vs)
             for lbt, ls, qp in shares(bt, L, 5, bounds)]
    o, lse = oracle.merge_lse([p[0] for p in parts], [p[1] for p in parts])
    full = oracle.paged_attention(q, pool, bt, L, 5, 2, ks, vs)
    assert np.allclose(o, full, rtol=1e-12, atol=1e-13)
    whole = oracle.paged_attention_partial(q, pool, bt, L, np.array(L) - 5, 5, 2, ks, vs)[1]
    assert np.allclose(lse, whole, rtol=0, atol=1e-12)


def test_rows_that_see_nothing():
    rng = np.random.default_rng(23)
    q, pool, bt, L, ks, vs = _random_case(rng, [20], 1, 2, 8, 5, 1)
    o, lse = oracle.paged_attention_partial(q, pool, bt, L, np.array([-10]), 5, 1, ks, vs)
    assert (o == 0).all() and np.isneginf(lse).all()
    o2, lse2 = oracle.merge_lse([o, o], [lse, lse])
    assert (o2 == 0).all() and np.isneginf(lse2).all()


def test_merge_against_scipy_logsumexp():
    rng = np.random.default_rng(24)
    po = rng.normal(size=(3, 7, 5, 16))
    pl = rng.normal(scale=30, size=(3, 7, 5))
    pl[1, 2, 3] = -np.inf
    o, lse = oracle.merge_lse(po, pl)
    want_lse = logsumexp(pl, axis=0)
    w = np.exp(pl - want_lse[None])
    assert np.allclose(lse, want_lse, rtol=0, atol=1e-12)
    assert np.allclose(o, np.einsum("prh,prhd->rhd", w, po), rtol=1e-12, atol=1e-12)
