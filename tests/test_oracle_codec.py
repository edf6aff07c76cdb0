"""Pins for the oracle's E4M3 / INT8 codecs and its quantize step.

Each pin checks the oracle against something other than itself: the values the
OCP OFP8 specification tabulates, torch's float8_e4m3fn type (an independent
library implementation), Python's built-in round-half-even, and brute-force
nearest-value search over the 254 finite codes.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ofp8_e4m3_special_values.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        lines = f.readlines()
    for line in lines:
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, bits, val = line.split()
        code = int(bits.replace(".", ""), 2)
        rows.append((name, code, float(val)))
    return rows


def test_golden_special_values_decode():
    rows = _golden_rows()
    assert len(rows) == 10
    for name, code, val in rows:
        got = float(oracle.e4m3_decode(code))
        if math.isnan(val):
            assert math.isnan(got), name
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), name


def test_golden_special_values_encode():
    for name, code, val in _golden_rows():
        if not math.isnan(val):
            assert int(oracle.e4m3_encode(val)) == code, name


def test_decode_all_codes_matches_torch_float8():
    codes = np.arange(256)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(got, ref, equal_nan=True)
    # signs of the two zeros too
    assert np.array_equal(np.signbit(got[[0, 0x80]]), [False, True])


def test_decode_monotone_and_symmetric():
    pos = oracle.e4m3_decode(np.arange(0, 0x7F))
    assert np.all(np.diff(pos) > 0)
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF))
    assert np.array_equal(neg, -pos)


def test_encode_decode_roundtrip_all_finite_codes():
    fin = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(fin)), fin.astype(np.uint8))


def _brute_e4m3(v):
    """Nearest finite E4M3 value by exhaustive search; ties -> even code;
    |v| > 448 -> +-448; the sign of zero follows v."""
    mags = oracle.e4m3_decode(np.arange(0, 0x7F))      # codes 0..126, increasing
    a = np.abs(v)
    dist = np.abs(a[:, None] - mags[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among equal-distance candidates (a tie between two neighbours) take the even code
    even = cand & (np.arange(0x7F)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    pick = np.where(a > 448.0, 0x7E, pick)
    return np.where(np.signbit(v), pick | 0x80, pick).astype(np.uint8)


@pytest.mark.parametrize("scale", [1.0, 86.625 / 448.0, 2.0 ** -7, 3.0, 1000.0])
def test_encode_matches_brute_force_over_all_fp16(scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x16 = bits.view(np.float16)
    x16 = x16[np.isfinite(x16)]
    v = codec.scaled_input(x16, scale)
    got = oracle.e4m3_encode(v)
    for a in range(0, len(v), 8192):
        sl = slice(a, a + 8192)
        assert np.array_equal(got[sl], _brute_e4m3(v[sl]))


@pytest.mark.parametrize("scale", [1.0, 86.625 / 448.0, 0.01])
def test_encode_matches_torch_cast_in_range(scale):
    # torch's cast rounds to nearest-even but maps overflow to NaN, so compare
    # only where the value does not exceed the largest finite code
    x16 = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    x16 = x16[np.isfinite(x16)]
    v = codec.scaled_input(x16, scale)
    keep = np.abs(v) <= 448.0
    ref = torch.from_numpy(v[keep].astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(oracle.e4m3_encode(v[keep]), ref.view(torch.uint8).numpy())


def test_encode_spot_values():
    cases = {448.0: 0x7E, 464.0: 0x7E, 480.0: 0x7E, 1e6: 0x7E, -1e6: 0xFE,
             2.0 ** -9: 0x01, 2.0 ** -10: 0x00, 1.5 * 2.0 ** -10: 0x01,
             2.5 * 2.0 ** -9: 0x02, 3.5 * 2.0 ** -9: 0x04, -0.0: 0x80, -1e-30: 0x80,
             1.0: 0x38, 1.0625: 0x38, 1.1875: 0x3A, 240.0: 0x77, 248.0: 0x78,
             float("inf"): 0x7E, float("-inf"): 0xFE, float("nan"): 0x7F}
    for x, c in cases.items():
        assert int(oracle.e4m3_encode(x)) == c, x


def test_int8_encode_vs_python_round():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(0, 60, 20000), np.arange(-300, 300) + 0.5,
                        np.arange(-140, 140, 0.25)])
    ref = np.array([max(-127, min(127, round(float(t)))) for t in x])
    assert np.array_equal(oracle.int8_encode(x), ref)


def test_int8_spot_values():
    x = [2.5, 3.5, -2.5, -3.5, 127.49, 127.5, 128.0, -127.5, -200.0, 0.4999,
         float("inf"), float("-inf"), float("nan")]
    want = [2, 4, -2, -4, 127, 127, 127, -127, -127, 0, 127, -127, 0]
    assert oracle.int8_encode(x).tolist() == want


def test_scaled_input_is_correctly_rounded_fp32_quotient():
    # compare with exact rational arithmetic for a random sample
    from fractions import Fraction
    rng = np.random.default_rng(3)
    xs = rng.normal(0, 10, 300).astype(np.float16)
    for s in [0.193359375, np.float32(86.625 / 448.0), np.float32(1.0 / 3.0)]:
        got = codec.scaled_input(xs, s)
        for x, g in zip(xs, got):
            exact = Fraction(float(x)) / Fraction(float(np.float32(s)))
            # nearest float32 to the exact quotient
            f = np.float32(float(exact))
            lo, hi = np.nextafter(f, np.float32(-np.inf)), np.nextafter(f, np.float32(np.inf))
            best = min([lo, f, hi], key=lambda c: (abs(Fraction(float(c)) - exact),
                                                   int(np.float32(c).view(np.uint32)) & 1))
            assert np.float32(g) == best


def test_quantize_fp16_is_identity_bits():
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    assert np.array_equal(oracle.quantize(x.view(np.float16), 1.0, 0), x)


def test_dequantize_int8_scale():
    c = np.array([-127, -1, 0, 1, 127], dtype=np.int8).view(np.uint8)
    assert np.array_equal(oracle.dequantize(c, 0.5, 2), [-63.5, -0.5, 0.0, 0.5, 63.5])
