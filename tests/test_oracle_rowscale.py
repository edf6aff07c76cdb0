"""Pins for format 3 (INT8 with a scale per (token, kv-head) row).

Pinned against things outside the oracle's own formula: the INT8 codec with
one scale (itself pinned in test_oracle_codec.py), exact rational arithmetic
for the scale's rounding to binary16, the properties round-half-even encoding must have
when no clamp is active, a per-key brute-force loop that reads the scale at
each slot, constant V, and the reduction to format 2 when every row has the
same largest value.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import attention as oatt

T3 = oracle.INT8_TOKEN


def _rows(rng, n, D=128, outliers=True):
    x = rng.normal(0, 1, (n, D)) * np.where(rng.random((n, D)) < 0.02, 20, 1)
    return x.astype(np.float16)


@pytest.mark.parametrize("amp", [1.0, 1e-3, 1e-6])     # 1e-6: scales below fp16's normal range
def test_scale_is_correctly_rounded_amax_over_127(amp):
    rng = np.random.default_rng(1)
    x = (_rows(rng, 300).astype(np.float32) * amp).astype(np.float16)
    s = oracle.int8_row_scale(x)
    for r in range(x.shape[0]):
        amax = Fraction(max(abs(float(e)) for e in x[r]))
        exact = amax / 127
        h = np.float16(s[r])
        assert float(h) == float(s[r])                   # a binary16 value
        got = Fraction(float(h))
        # the nearest binary16 to amax/127 (ties to even): no other fp16 is closer
        up = Fraction(float(np.nextafter(h, np.float16(np.inf))))
        dn = Fraction(float(np.nextafter(h, np.float16(0))))
        assert abs(got - exact) <= abs(up - exact) and abs(got - exact) <= abs(dn - exact)
        if abs(got - exact) == abs(up - exact) or (got != 0 and abs(got - exact) == abs(dn - exact)):
            assert (h.view(np.uint16) & 1) == 0


def test_row_codes_equal_int8_codec_with_that_rows_scale():
    rng = np.random.default_rng(2)
    x = _rows(rng, 64)
    s = oracle.int8_row_scale(x)
    got = oracle.quantize(x, s, T3)
    for r in range(x.shape[0]):
        assert np.array_equal(got[r], oracle.quantize(x[r], s[r], 2))


def test_largest_element_gets_127_and_error_is_half_a_step():
    rng = np.random.default_rng(3)
    x = _rows(rng, 200)
    s = oracle.int8_row_scale(x).astype(np.float64)
    c = oracle.quantize(x, oracle.int8_row_scale(x), T3).view(np.int8).astype(np.int64)
    xf = x.astype(np.float64)
    for r in range(x.shape[0]):
        j = int(np.argmax(np.abs(xf[r])))
        assert abs(c[r, j]) == 127 and np.sign(c[r, j]) == np.sign(xf[r, j])
        assert np.abs(c[r]).max() == 127
        err = np.abs(xf[r] - c[r] * s[r])
        assert (err <= s[r] * (0.5 + 2.0 ** -20)).all()


def test_zero_and_nan_rows():
    x = np.zeros((3, 8), dtype=np.float16)
    x[1, 3] = np.nan
    x[1, 5] = -2.0
    x[2, :] = np.nan
    s = oracle.int8_row_scale(x)
    assert s[0] == 0 and s[2] == 0 and s[1] == np.float32(np.float16(2.0 / 127))
    c = oracle.quantize(x, s, T3).view(np.int8)
    assert (c[0] == 0).all() and (c[2] == 0).all()
    assert c[1, 3] == 0 and c[1, 5] == -127


def _case3(rng, L, H, G, D, q_len, P=16):
    B = len(L)
    need = [(x + P - 1) // P for x in L]
    num_pages = sum(need) + 2
    perm = rng.permutation(num_pages)
    bt = np.full((B, max(need)), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    pool = oracle.new_pool(num_pages, H, D, T3, P)
    kp = oracle.new_scale_pool(num_pages, H, P)
    vp = oracle.new_scale_pool(num_pages, H, P)
    for s in range(B):
        k = _rows(rng, L[s] * H, D).reshape(L[s], H, D)
        v = _rows(rng, L[s] * H, D).reshape(L[s], H, D) * np.float16(0.5)
        t = np.arange(L[s])
        slots = bt[s, t // P].astype(np.int64) * P + t % P
        pool, kp, vp = oracle.kv_append_quant(k, v, slots, T3, kp, vp, pool)
    q = rng.normal(0, 1, (B * q_len, H * G, D)).astype(np.float16)
    return q, pool, bt, np.array(L), kp, vp


def _brute3(q, pool, bt, L, q_len, kp, vp):
    """Per-key loop reading each row's scale at its slot."""
    BQ, Hq, D = q.shape
    H = pool.shape[1]
    G = Hq // H
    P = pool.shape[3]
    out = np.zeros((BQ, Hq, D))
    for s in range(len(L)):
        for i in range(q_len):
            pos = L[s] - q_len + i
            for hq in range(Hq):
                h = hq // G
                qv = [float(x) for x in q[s * q_len + i, hq]]
                scores, vals = [], []
                for j in range(pos + 1):
                    page, off = bt[s, j // P], j % P
                    kc = pool[page, h, 0, off].view(np.int8)
                    vc = pool[page, h, 1, off].view(np.int8)
                    ks, vs = float(kp[page, h, off]), float(vp[page, h, off])
                    dot = math.fsum(qv[d] * int(kc[d]) * ks for d in range(D))
                    scores.append(dot / math.sqrt(D))
                    vals.append([int(c) * vs for c in vc])
                mx = max(scores)
                w = [math.exp(x - mx) for x in scores]
                tot = math.fsum(w)
                for d in range(D):
                    out[s * q_len + i, hq, d] = math.fsum(w[j] * vals[j][d] for j in range(len(w))) / tot
    return out


@pytest.mark.parametrize("q_len,G", [(1, 4), (5, 2)])
def test_brute_force_tiny_row_scaled(q_len, G):
    rng = np.random.default_rng(40 + q_len)
    q, pool, bt, L, kp, vp = _case3(rng, [7, 21, 34], 2, G, 8, q_len)
    got = oracle.paged_attention(q, pool, bt, L, q_len, T3, kp, vp)
    ref = _brute3(q, pool, bt, L, q_len, kp, vp)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_constant_v_rows_give_that_row():
    rng = np.random.default_rng(7)
    q, pool, bt, L, kp, vp = _case3(rng, [40, 9], 2, 4, 16, 5)
    row = np.linspace(-3, 3, 16).astype(np.float16)
    s = oracle.int8_row_scale(row[None])[0]
    codes = oracle.quantize(row[None], np.array([s]), T3)[0]
    pool[:, :, 1] = codes
    vp[:] = s
    want = codes.view(np.int8).astype(np.float64) * float(s)
    got = oracle.paged_attention(q, pool, bt, L, 5, T3, kp, vp)
    assert np.allclose(got, np.broadcast_to(want, got.shape), rtol=1e-14, atol=0)


def test_equal_row_maxima_reduce_to_one_scale_int8():
    # every row holds +-A somewhere, so every row's scale is A/127: format 3
    # must then give exactly what format 2 gives with that single scale
    rng = np.random.default_rng(9)
    L, H, D, P = [30], 1, 16, 16
    A = np.float16(6.0)
    k = rng.uniform(-5, 5, (L[0], H, D)).astype(np.float16)
    v = rng.uniform(-5, 5, (L[0], H, D)).astype(np.float16)
    k[np.arange(L[0]), 0, rng.integers(0, D, L[0])] = A
    v[np.arange(L[0]), 0, rng.integers(0, D, L[0])] = -A
    n = 2
    bt = np.array([[1, 0]], dtype=np.int32)
    t = np.arange(L[0])
    slots = bt[0, t // P].astype(np.int64) * P + t % P
    p3, kp, vp = oracle.kv_append_quant(k, v, slots, T3, oracle.new_scale_pool(n, H, P),
                                        oracle.new_scale_pool(n, H, P), oracle.new_pool(n, H, D, T3))
    s = np.float32(np.float16(float(A) / 127))          # the row scale, a binary16 value
    p2 = oracle.kv_append_quant(k, v, slots, 2, [s], [s], oracle.new_pool(n, H, D, 2))
    assert np.array_equal(p3, p2)
    q = rng.normal(0, 1, (5, 2, D)).astype(np.float16)
    a = oracle.paged_attention(q, p3, bt, L, 5, T3, kp, vp)
    b = oracle.paged_attention(q, p2, bt, L, 5, 2, [s], [s])
    assert np.array_equal(a, b)


def test_planted_wrong_axis_is_caught(monkeypatch):
    # a scale taken over the wrong axis (per column instead of per row) must
    # fail the largest-element pin
    bad = lambda x16: (np.abs(np.asarray(x16, np.float16).astype(np.float64)).max(axis=0)
                       / 127).astype(np.float32)[: np.asarray(x16).shape[0]]
    rng = np.random.default_rng(3)
    x = _rows(rng, 128)
    s = bad(x)
    c = oracle.quantize(x, s, T3).view(np.int8).astype(np.int64)
    assert any(np.abs(c[r]).max() != 127 for r in range(x.shape[0]))
