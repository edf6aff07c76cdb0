"""Oracle: E4M3 and INT8 KV codes, written from their definitions.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg use it.

Formats
-------
* FP8 E4M3 is the "FN" variant of the OCP 8-bit floating point specification
  (OFP8, rev. 1.0): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
  infinities, NaN = S.1111.111, largest finite value 448.  The ReVolta README
  ("Weight and KV formats", "E4M3 KV") stores the KV cache in this format with
  calibrated per-layer K and V scales; a scale equal to amax / 448 maps the
  layer's largest value to the largest finite code.
* INT8 is symmetric: code = clamp(round_half_even(x), -127, 127), value =
  code * scale (ReVolta README, "Weight and KV formats", "INT8 KV").
* INT8 with a scale per row (format 3): the same codes, but every (token,
  kv-head) row of K and of V carries its own scale, computed when the row is
  written -- the README's INT8 KV, whose scales come from the data at run time
  for each token and head instead of from a calibration.  The scale is the
  row's largest |x| (NaNs ignored; 0 for a row of zeros) divided by 127,
  rounded once to binary32; each element is then encoded as above under it.

Rounding is to nearest with ties to even everywhere; encoding saturates.
For non-finite inputs the oracle takes the reading that E4M3 maps NaN to the
NaN code 0x7F and +-Inf to +-448, and INT8 maps NaN to 0 and +-Inf to +-127
(parity unpinned by the pages, which never feed such values).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
INT8_MAX = 127
INT8_TOKEN = 3          # kv format code: INT8 with a scale per (token, kv-head) row


def e4m3_decode(codes) -> np.ndarray:
    """Real value of each E4M3 code, float64 (NaN for 0x7F / 0xFF).

    code = s*2^7 + e*2^3 + m:  e = 0 gives (-1)^s * 2^-6 * m/8,
    1 <= e <= 15 gives (-1)^s * 2^(e-7) * (1 + m/8), e = 15 with m = 7 is NaN.
    """
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 code (uint8) nearest to each real x, ties to the even code,
    saturating at +-448; zero keeps the sign of x; NaN -> 0x7F.

    The magnitude code is built as (biased exponent << 3) + rounded mantissa,
    so a mantissa that rounds up to 8 carries into the exponent field, which is
    exactly the next binade's first value.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # everything above 464 saturates; clamping keeps +-Inf out of the arithmetic
    a = np.minimum(a, 1024.0)
    # exponent of the binade holding a, clamped to the normal range [-6, 8]
    with np.errstate(divide="ignore"):
        ex = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # guard against log2 being off by one at exact powers of two
    ex = np.where(np.ldexp(1.0, ex.astype(np.int64)) > a, ex - 1, ex)
    ex = np.where(np.ldexp(1.0, (ex + 1).astype(np.int64)) <= a, ex + 1, ex)
    ex = np.clip(ex, -6, 8).astype(np.int64)
    # quantum of that binade: 2^(ex - 3); subnormals share the -6 binade quantum
    q = np.rint(np.ldexp(a, -(ex - 3)))           # round half to even
    # q counts multiples of the quantum: q in [8, 16] for normals, [0, 8] below
    biased = np.where(a >= 2.0 ** -6, ex + 7, 0)
    mag = np.where(biased == 0, q, (biased << 3) + (q - 8)).astype(np.int64)
    mag = np.minimum(mag, 0x7E)                   # saturate at 448
    mag = np.where(nan, 0x7F, mag)
    code = np.where(sign & ~nan, mag | 0x80, mag)
    return code.astype(np.uint8)


def int8_encode(x) -> np.ndarray:
    """INT8 code: round half to even, clamp to [-127, 127]; NaN -> 0."""
    x = np.asarray(x, dtype=np.float64)
    r = np.rint(np.nan_to_num(x, nan=0.0, posinf=1e30, neginf=-1e30))
    return np.clip(r, -INT8_MAX, INT8_MAX).astype(np.int8)


def int8_decode(codes) -> np.ndarray:
    return np.asarray(codes).astype(np.int8).astype(np.float64)


def scaled_input(x16, scale) -> np.ndarray:
    """The value that gets encoded: fp32(x) / fp32(scale) as a correctly rounded
    binary32 quotient.  The quotient is formed in float64 and rounded once to
    float32; double rounding is innocuous for division since 53 >= 2*24 + 2
    (Figueroa, "When is double rounding innocuous?", 1995)."""
    xf = np.asarray(x16).astype(np.float32).astype(np.float64)
    sf = np.asarray(scale, dtype=np.float32).astype(np.float64)
    return (xf / sf).astype(np.float32).astype(np.float64)


def int8_row_scale(x16) -> np.ndarray:
    """Scale of each row (last axis) of fp16 values for format 3, a binary16
    value (returned as float32, which holds it exactly): fp16(amax / 127),
    amax = the row's largest |x| with NaNs ignored (0 when nothing else is
    left).  The quotient is formed in float64 and rounded once more to fp16;
    double rounding is innocuous for division since 53 >= 2*11 + 2."""
    a = np.abs(np.asarray(x16, dtype=np.float16).astype(np.float64))
    a = np.where(np.isnan(a), 0.0, a)
    return (a.max(axis=-1) / INT8_MAX).astype(np.float16).astype(np.float32)


def quantize(x16, scale, kv_dtype: int) -> np.ndarray:
    """Codes stored in the pool for fp16 inputs x16 under ``scale``.

    kv_dtype 0 (FP16): the fp16 bits unchanged (uint16 view); 1 (E4M3): uint8
    codes; 2 (INT8): int8 codes viewed as uint8.
    """
    x16 = np.asarray(x16, dtype=np.float16)
    if kv_dtype == 0:
        return x16.view(np.uint16).copy()
    if kv_dtype == INT8_TOKEN:
        # ``scale`` holds one value per row (the leading axes of x16)
        scale = np.asarray(scale, dtype=np.float32)[..., None]
    with np.errstate(invalid="ignore", divide="ignore"):
        v = scaled_input(x16, scale)          # a zero scale leaves 0/0 = NaN -> code 0
    if kv_dtype == 1:
        return e4m3_encode(v)
    if kv_dtype in (2, INT8_TOKEN):
        return int8_encode(v).view(np.uint8)
    raise ValueError(kv_dtype)


def dequantize(codes, scale, kv_dtype: int) -> np.ndarray:
    """float64 value of stored codes (exact: code value times the scale)."""
    codes = np.asarray(codes)
    if kv_dtype == 0:
        return codes.astype(np.uint16).view(np.float16).astype(np.float64)
    s = np.asarray(scale, dtype=np.float32).astype(np.float64)
    if kv_dtype == 1:
        return e4m3_decode(codes.astype(np.uint8)) * s
    if kv_dtype == 2:
        return int8_decode(codes.astype(np.uint8).view(np.int8)) * s
    if kv_dtype == INT8_TOKEN:
        return int8_decode(codes.astype(np.uint8).view(np.int8)) * s[..., None]
    raise ValueError(kv_dtype)
