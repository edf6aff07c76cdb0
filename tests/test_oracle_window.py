"""Pins for the oracle's sliding-window attention (ReVolta README, "DFlash2
speculative decoding": sliding-window layers with a 2048-token window; the
reading taken: query position p sees keys p - window + 1 .. p).

Independent of the oracle's vectorised code: a per-query loop with Python's
math module over exactly the keys in the window, the exact reductions
(a window of one key returns that key's V; a window as long as the cache is
plain causal attention), and the identity with a cache truncated to the
window's keys.  A planted off-by-one in the window bound trips the loop pin.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import attention as oatt
from tests.test_oracle_attention import _decode_code, _random_case


def _brute_window(q, pool, bt, L, q_len, kv_dtype, ks, vs, window):
    BQ, Hq, D = q.shape
    H = pool.shape[1]
    G = Hq // H
    P = pool.shape[3]
    out = np.zeros((BQ, Hq, D))
    for s in range(len(L)):
        for i in range(q_len):
            pos = L[s] - q_len + i
            lo = max(0, pos - window + 1)
            for hq in range(Hq):
                h = hq // G
                ksc = float(ks[h % len(ks)]) if kv_dtype else 1.0
                vsc = float(vs[h % len(vs)]) if kv_dtype else 1.0
                qv = [float(x) for x in q[s * q_len + i, hq]]
                scores, vals = [], []
                for j in range(lo, pos + 1):
                    page = bt[s, j // P]
                    krow, vrow = pool[page, h, 0, j % P], pool[page, h, 1, j % P]
                    dot = math.fsum(qv[d] * _decode_code(int(krow[d]), kv_dtype) * ksc
                                    for d in range(D))
                    scores.append(dot / math.sqrt(D))
                    vals.append([_decode_code(int(x), kv_dtype) * vsc for x in vrow])
                mx = max(scores)
                w = [math.exp(x - mx) for x in scores]
                tot = math.fsum(w)
                for d in range(D):
                    out[s * q_len + i, hq, d] = math.fsum(
                        w[j] * vals[j][d] for j in range(len(w))) / tot
    return out


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("window", [1, 3, 16, 17, 30])
def test_window_matches_per_key_loop(kv_dtype, window):
    rng = np.random.default_rng(700 + 10 * kv_dtype + window)
    q_len, G = 5, 2
    q, pool, bt, L, ks, vs = _random_case(rng, [7, 19, 41], 2, G, 8, q_len, kv_dtype,
                                          scale_per_head=(kv_dtype == 2))
    got = oracle.paged_attention(q, pool, bt, L, q_len, kv_dtype, ks, vs, window=window)
    ref = _brute_window(q, pool, bt, L, q_len, kv_dtype, ks, vs, window)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_window_of_one_returns_own_value():
    """A single visible key: the softmax weight is exactly 1."""
    rng = np.random.default_rng(71)
    q_len, G = 5, 4
    q, pool, bt, L, ks, vs = _random_case(rng, [23, 40], 2, G, 16, q_len, 1)
    got = oracle.paged_attention(q, pool, bt, L, q_len, 1, ks, vs, window=1)
    for s, Ls in enumerate(L):
        for h in range(2):
            _, V = oracle.gather_kv(pool, bt[s], Ls, h, 1, ks[0], vs[0])
            for i in range(q_len):
                own = V[Ls - q_len + i]
                for g in range(G):
                    assert np.array_equal(got[s * q_len + i, h * G + g], own)


@pytest.mark.parametrize("window", [0, 41, 1000])
def test_window_as_long_as_the_cache_is_causal_attention(window):
    rng = np.random.default_rng(72)
    q, pool, bt, L, ks, vs = _random_case(rng, [41, 12], 2, 4, 16, 5, 2)
    full = oracle.paged_attention(q, pool, bt, L, 5, 2, ks, vs)
    got = oracle.paged_attention(q, pool, bt, L, 5, 2, ks, vs, window=window)
    assert np.array_equal(got, full)


def test_window_one_short_hides_only_the_first_key_from_the_last_row():
    """L = 41, window 40: the last query (position 40) no longer sees key 0;
    the earlier four rows still see every key they may see."""
    rng = np.random.default_rng(72)
    q, pool, bt, L, ks, vs = _random_case(rng, [41, 12], 2, 4, 16, 5, 2)
    full = oracle.paged_attention(q, pool, bt, L, 5, 2, ks, vs)
    got = oracle.paged_attention(q, pool, bt, L, 5, 2, ks, vs, window=40)
    assert np.array_equal(got[:4], full[:4])                 # sequence 0, queries 0-3
    assert not np.allclose(got[4], full[4])                  # sequence 0, query 4
    assert np.array_equal(got[5:], full[5:])                 # sequence 1 (12 <= 40)


@pytest.mark.parametrize("window", [5, 16, 21])
def test_window_equals_cache_truncated_to_the_window(window):
    """q_len 1: the window's result equals plain attention over a cache that
    holds only the window's keys (no positional term enters the scores)."""
    rng = np.random.default_rng(73 + window)
    q, pool, bt, L, ks, vs = _random_case(rng, [45], 1, 4, 16, 1, 1)
    got = oracle.paged_attention(q, pool, bt, L, 1, 1, ks, vs, window=window)
    Ls = int(L[0])
    lo = Ls - window
    # re-page the window's keys into a fresh pool at positions 0 .. window-1
    n = (window + 15) // 16
    pool2 = oracle.new_pool(n, 1, 16, 1)
    for j in range(lo, Ls):
        src = pool[bt[0, j // 16], 0, :, j % 16]
        pool2[(j - lo) // 16, 0, :, (j - lo) % 16] = src
    bt2 = np.arange(n, dtype=np.int32)[None, :]
    ref = oracle.paged_attention(q, pool2, bt2, [window], 1, 1, ks, vs)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_planted_off_by_one_window_is_caught(monkeypatch):
    rng = np.random.default_rng(74)
    q, pool, bt, L, ks, vs = _random_case(rng, [33], 2, 2, 8, 5, 1)
    ref = _brute_window(q, pool, bt, L, 5, 1, ks, vs, 9)
    real = oatt.attention_partial

    def off_by_one(qrows, K, V, limits, j0, j1, lower=None):
        return real(qrows, K, V, limits, j0, j1, None if lower is None else lower - 1)

    monkeypatch.setattr(oatt, "attention_partial", off_by_one)
    bad = oracle.paged_attention(q, pool, bt, L, 5, 1, ks, vs, window=9)
    assert not np.allclose(bad, ref, rtol=1e-9, atol=1e-12)
