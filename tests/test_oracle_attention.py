"""Pins for the oracle's append, paged attention and split-KV merge.

The pins are independent of the oracle's own code path: a per-query loop with
Python's math module and torch's float8 decode (brute force on tiny inputs),
torch's scaled_dot_product_attention in float64 (unpaged reduction), and exact
identities of the definition (constant V, page-order, split count, causal
truncation, GQA == MHA with repeated K/V).  The last test plants plausible
mistakes in the oracle and checks that some pin catches each.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oatt


def _random_case(rng, L, H, G, D, q_len, kv_dtype, P=16, slack=3, scale_per_head=False):
    B = len(L)
    need = [(x + P - 1) // P for x in L]
    num_pages = sum(need) + slack
    perm = rng.permutation(num_pages)
    bt = np.full((B, max(need)), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    pool = oracle.new_pool(num_pages, H, D, kv_dtype, P)
    nsc = H if scale_per_head else 1
    ks = rng.uniform(0.05, 0.3, nsc).astype(np.float32)
    vs = rng.uniform(0.05, 0.3, nsc).astype(np.float32)
    for s in range(B):
        k = (rng.normal(0, 1, (L[s], H, D)) * np.where(rng.random((L[s], H, D)) < 0.05, 20, 1))
        v = rng.normal(0, 1, (L[s], H, D))
        t = np.arange(L[s])
        slots = bt[s, t // P].astype(np.int64) * P + t % P
        pool = oracle.kv_append_quant(k.astype(np.float16), v.astype(np.float16), slots,
                                      kv_dtype, ks, vs, pool)
    q = rng.normal(0, 1, (B * q_len, H * G, D)).astype(np.float16)
    return q, pool, bt, np.array(L), ks, vs


def _decode_code(c, kv_dtype):
    # independent decode: torch's float8 type / int8 / fp16 bit reinterpretation
    if kv_dtype == 0:
        return float(np.array([c], dtype=np.uint16).view(np.float16)[0])
    if kv_dtype == 1:
        return float(torch.tensor([int(c)], dtype=torch.uint8).view(torch.float8_e4m3fn).double())
    return float(np.array([c], dtype=np.uint8).view(np.int8)[0])


def _brute(q, pool, bt, L, q_len, kv_dtype, ks, vs):
    """Per-query loop: every score and weight is formed one key at a time."""
    BQ, Hq, D = q.shape
    H = pool.shape[1]
    G = Hq // H
    P = pool.shape[3]
    out = np.zeros((BQ, Hq, D))
    cache = {}

    def dec(c):
        if c not in cache:
            cache[c] = _decode_code(c, kv_dtype)
        return cache[c]

    for s in range(len(L)):
        for i in range(q_len):
            pos = L[s] - q_len + i
            for hq in range(Hq):
                h = hq // G
                ksc = float(ks[h % len(ks)]) if kv_dtype else 1.0
                vsc = float(vs[h % len(vs)]) if kv_dtype else 1.0
                qv = [float(x) for x in q[s * q_len + i, hq]]
                scores = []
                vals = []
                for j in range(pos + 1):
                    page = bt[s, j // P]
                    krow = pool[page, h, 0, j % P]
                    vrow = pool[page, h, 1, j % P]
                    dot = 0.0
                    for d in range(D):
                        dot += qv[d] * dec(int(krow[d])) * ksc
                    scores.append(dot / math.sqrt(D))
                    vals.append([dec(int(x)) * vsc for x in vrow])
                mx = max(scores)
                w = [math.exp(x - mx) for x in scores]
                tot = math.fsum(w)
                for d in range(D):
                    out[s * q_len + i, hq, d] = math.fsum(w[j] * vals[j][d] for j in range(len(w))) / tot
    return out


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("q_len,G", [(1, 1), (5, 2), (1, 4)])
def test_brute_force_tiny(kv_dtype, q_len, G):
    rng = np.random.default_rng(100 + 10 * kv_dtype + q_len + G)
    L = [7, 19, 33]
    D = 8
    q, pool, bt, L, ks, vs = _random_case(rng, L, 2, G, D, q_len, kv_dtype,
                                          scale_per_head=(kv_dtype == 2))
    got = oracle.paged_attention(q, pool, bt, L, q_len, kv_dtype, ks, vs)
    ref = _brute(q, pool, bt, L, q_len, kv_dtype, ks, vs)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_brute_force_full_head_dim():
    rng = np.random.default_rng(5)
    q, pool, bt, L, ks, vs = _random_case(rng, [21], 1, 2, 128, 5, 1)
    got = oracle.paged_attention(q, pool, bt, L, 5, 1, ks, vs)
    ref = _brute(q, pool, bt, L, 5, 1, ks, vs)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kv_dtype,code,scale", [(1, 0x3A, 0.25), (1, 0xC9, 0.125),
                                                  (2, 0x85, 0.5), (0, 0x3C00, 1.0)])
def test_constant_v_gives_that_constant(kv_dtype, code, scale):
    rng = np.random.default_rng(11)
    q, pool, bt, L, ks, vs = _random_case(rng, [40, 9], 2, 4, 16, 5, kv_dtype)
    pool[:, :, 1] = code
    vs = np.array([scale], dtype=np.float32)
    want = oracle.dequantize(np.array([code]), scale, kv_dtype)[0]
    got = oracle.paged_attention(q, pool, bt, L, 5, kv_dtype, ks, vs)
    assert np.allclose(got, want, rtol=1e-14, atol=0)


def test_page_order_invariance_is_bitwise():
    rng = np.random.default_rng(12)
    q, pool, bt, L, ks, vs = _random_case(rng, [50, 77, 16], 2, 4, 32, 5, 1, slack=9)
    a = oracle.paged_attention(q, pool, bt, L, 5, 1, ks, vs)
    perm = rng.permutation(pool.shape[0])          # new_position -> old page
    inv = np.argsort(perm)                          # old page -> new position
    pool2 = pool[perm]
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    b = oracle.paged_attention(q, pool2, bt2, L, 5, 1, ks, vs)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("splits", [2, 3, 7, 64])
def test_split_invariance(splits):
    rng = np.random.default_rng(13)
    q, pool, bt, L, ks, vs = _random_case(rng, [300, 65, 130], 2, 4, 32, 5, 1)
    a = oracle.paged_attention(q, pool, bt, L, 5, 1, ks, vs, num_splits=1)
    b = oracle.paged_attention(q, pool, bt, L, 5, 1, ks, vs, num_splits=splits)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_unpaged_reduction_matches_torch_sdpa():
    # one page holding the whole sequence: the result must equal textbook
    # softmax(Q K^T / sqrt(D)) V on dense arrays with a causal mask inside q_len
    rng = np.random.default_rng(14)
    Lx, D, q_len, G = 37, 64, 5, 4
    q, pool, bt, L, ks, vs = _random_case(rng, [Lx], 1, G, D, q_len, 2, P=Lx, slack=0)
    got = oracle.paged_attention(q, pool, bt, L, q_len, 2, ks, vs)
    K = pool[bt[0, 0], 0, 0].view(np.int8).astype(np.float64) * float(ks[0])
    V = pool[bt[0, 0], 0, 1].view(np.int8).astype(np.float64) * float(vs[0])
    Q = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)          # [Hq, q_len, D]
    mask = torch.arange(Lx)[None, :] <= (Lx - q_len + torch.arange(q_len))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, torch.from_numpy(K)[None].expand(G, -1, -1), torch.from_numpy(V)[None].expand(G, -1, -1),
        attn_mask=mask)
    assert np.allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-14)


def test_causal_row_equals_truncated_decode():
    rng = np.random.default_rng(15)
    q_len = 5
    q, pool, bt, L, ks, vs = _random_case(rng, [45, 23], 2, 4, 16, q_len, 1)
    full = oracle.paged_attention(q, pool, bt, L, q_len, 1, ks, vs)
    for s in range(2):
        for i in range(q_len):
            qi = q[s * q_len + i][None]
            Li = np.array([L[s] - q_len + i + 1])
            one = oracle.paged_attention(qi, pool, bt[s:s + 1], Li, 1, 1, ks, vs)
            assert np.allclose(one[0], full[s * q_len + i], rtol=1e-13, atol=1e-15)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(16)
    G = 4
    q, pool, bt, L, ks, vs = _random_case(rng, [40, 18], 2, G, 16, 5, 2, scale_per_head=True)
    a = oracle.paged_attention(q, pool, bt, L, 5, 2, ks, vs)
    pool_mha = np.repeat(pool, G, axis=1)           # kv-head h -> q-heads h*G .. h*G+G-1
    b = oracle.paged_attention(q, pool_mha, bt, L, 5, 2, np.repeat(ks, G), np.repeat(vs, G))
    assert np.array_equal(a, b)


def test_lse_merge_of_two_halves_equals_softmax():
    rng = np.random.default_rng(17)
    K = rng.normal(0, 3, (50, 8))
    V = rng.normal(0, 1, (50, 8))
    qr = rng.normal(0, 1, (3, 8))
    lim = np.array([49, 49, 20])
    parts = [oatt.attention_partial(qr, K, V, lim, 0, 25), oatt.attention_partial(qr, K, V, lim, 25, 50)]
    got = oracle.lse_merge(parts)
    S = qr @ K.T / np.sqrt(8)
    S = np.where(np.arange(50)[None] <= lim[:, None], S, -np.inf)
    P = np.exp(S - S.max(1, keepdims=True))
    want = (P / P.sum(1, keepdims=True)) @ V
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14)
    # row 2 sees nothing of the second half: that partial must be empty
    assert parts[1][1][2] == -np.inf and parts[1][2][2] == 0.0


# ----------------------------------------------------------------------------
# append
# ----------------------------------------------------------------------------

def test_append_writes_only_target_slots_in_layout():
    rng = np.random.default_rng(18)
    H, D, P = 3, 16, 16
    pool = oracle.new_pool(10, H, D, 1, P, fill=0xAB)
    k = rng.normal(0, 1, (4, H, D)).astype(np.float16)
    v = rng.normal(0, 1, (4, H, D)).astype(np.float16)
    slots = np.array([37, -1, 5, 159])
    out = oracle.kv_append_quant(k, v, slots, 1, [0.5], [0.25], pool)
    changed = np.argwhere(out != pool)
    touched = {(int(p), int(o)) for p, _, _, o, _ in changed}
    assert touched <= {(2, 5), (0, 5), (9, 15)}
    for t, slot in [(0, 37), (2, 5), (3, 159)]:
        page, off = divmod(slot, P)
        for h in range(H):
            assert np.array_equal(out[page, h, 0, off], oracle.e4m3_encode(k[t, h].astype(np.float64) / 0.5))
            assert np.array_equal(out[page, h, 1, off], oracle.e4m3_encode(v[t, h].astype(np.float64) / 0.25))


def test_append_duplicate_slot_later_token_wins():
    pool = oracle.new_pool(2, 1, 4, 2, 16)
    k = np.array([[[1, 2, 3, 4]], [[5, 6, 7, 8]]], dtype=np.float16)
    out = oracle.kv_append_quant(k, k, [3, 3], 2, [1.0], [1.0], pool)
    assert out[0, 0, 0, 3].view(np.int8).tolist() == [5, 6, 7, 8]


def test_append_rejects_slot_outside_pool():
    pool = oracle.new_pool(2, 1, 4, 1, 16)
    k = np.zeros((1, 1, 4), dtype=np.float16)
    with pytest.raises(IndexError):
        oracle.kv_append_quant(k, k, [32], 1, [1.0], [1.0], pool)


# ----------------------------------------------------------------------------
# planted mistakes: each plausible bug must trip at least one pin above
# ----------------------------------------------------------------------------

def _pins_pass(fns):
    try:
        for f in fns:
            f()
    except AssertionError:
        return False
    return True


def test_planted_mistakes_are_caught(monkeypatch):
    pins = [lambda: test_brute_force_tiny(1, 5, 2), test_unpaged_reduction_matches_torch_sdpa,
            test_gqa_equals_mha_with_repeated_kv, test_causal_row_equals_truncated_decode,
            test_golden_like_decode]
    assert _pins_pass(pins)

    # 1. softmax scale 1/D instead of 1/sqrt(D)
    orig_partial = oatt.attention_partial

    def bad_scale(qrows, K, V, limits, j0, j1, lower=None):
        return orig_partial(qrows / np.sqrt(qrows.shape[1]), K, V, limits, j0, j1, lower)
    monkeypatch.setattr(oatt, "attention_partial", bad_scale)
    assert not _pins_pass(pins)
    monkeypatch.setattr(oatt, "attention_partial", orig_partial)

    # 2. causal limit off by one
    def bad_causal(qrows, K, V, limits, j0, j1, lower=None):
        return orig_partial(qrows, K, V, np.asarray(limits) + 1, j0, min(j1 + 1, K.shape[0]),
                            lower)
    monkeypatch.setattr(oatt, "attention_partial", bad_causal)
    assert not _pins_pass(pins)
    monkeypatch.setattr(oatt, "attention_partial", orig_partial)

    # 3. GQA mapping h = hq % Hkv instead of hq // G
    orig_rows = oatt._rows_of

    def bad_rows(q, s, h, q_len, G):
        q = np.asarray(q)
        H = q.shape[1] // G
        blk = q[s * q_len:(s + 1) * q_len, h::H].astype(np.float64)
        return blk.reshape(q_len * G, -1)
    monkeypatch.setattr(oatt, "_rows_of", bad_rows)
    assert not _pins_pass(pins)
    monkeypatch.setattr(oatt, "_rows_of", orig_rows)

    # 4. E4M3 exponent bias 8 instead of 7
    from oracle import codec
    orig_dec = codec.e4m3_decode
    monkeypatch.setattr(codec, "e4m3_decode", lambda c: orig_dec(c) * 0.5)
    monkeypatch.setattr(oracle, "e4m3_decode", codec.e4m3_decode)
    assert not _pins_pass(pins)


def test_golden_like_decode():
    # OFP8 largest finite value and smallest subnormal (see tests/golden)
    from oracle import codec
    assert codec.e4m3_decode(0x7E) == 448.0 and codec.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.dequantize(np.array([0x7E]), 1.0, 1)[0] == 448.0
